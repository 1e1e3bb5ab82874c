"""Thin ctypes binding of libnsv.so (declared in include/nsv.h).

Argument marshalling only: every step of the decode read and the KV append
runs in the library's CUDA kernels.  Tensors are torch tensors on the current
CUDA device, C-contiguous, in the layouts nsv.h documents:

  q, out          [rows, num_heads, head_dim]               float32 | bfloat16
                  or [rows, query_len, num_heads, head_dim] (several query
                  tokens per row, causal among themselves)
  k_pool, v_pool  [num_blocks + 1, num_kv_heads, 16, head_dim]  (last = sink)
  k_new, v_new    [rows, num_kv_heads, head_dim] or [rows, query_len, ...]
  write_slots     [rows] or [rows, query_len] int64
  block_tables    [rows, max_blocks] int32
  context_lens    [rows] int32

Importing this module loads the library and raises ImportError if it has not
been built (``python -m paged_kv_decode_nsv_gb300.build``); there is no
fallback path.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libnsv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libnsv.so is not built (%s); run python -m paged_kv_decode_nsv_gb300.build"
                      % LIB_PATH)

_lib = ctypes.CDLL(LIB_PATH)

ABI_VERSION = 102  # the layout of Shape and Plan below
F32, BF16 = 0, 1
(CONSUMER_AUTO, CONSUMER_CUDA, CONSUMER_TENSOR, CONSUMER_TENSOR_VECTOR_ROWS,
 CONSUMER_TENSOR_TMEM) = 0, 1, 2, 3, 4
DEV_BAD_CTX, DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_TIMEOUT = 1, 2, 4, 8
ERRORS = {0: "NSV_OK", -1: "NSV_ERR_NULLPTR", -2: "NSV_ERR_DTYPE", -3: "NSV_ERR_SHAPE",
          -4: "NSV_ERR_ALIGN", -5: "NSV_ERR_RANGE", -6: "NSV_ERR_CAPTURE", -7: "NSV_ERR_CUDA",
          -8: "NSV_ERR_WORKSPACE", -10: "NSV_ERR_UNSUPPORTED"}


class Shape(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("query_len", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("kv_heads_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("vectors_per_warp", ctypes.c_int32),
                ("consumer", ctypes.c_int32), ("blocks_per_stage", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_vp, _i32, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_SP, _PP = ctypes.POINTER(Shape), ctypes.POINTER(Plan)

_lib.nsv_abi_version.restype = _i32
_lib.nsv_abi_version.argtypes = []
if _lib.nsv_abi_version() != ABI_VERSION:
    raise ImportError("libnsv.so has ABI version %d, this binding expects %d; rebuild it"
                      % (_lib.nsv_abi_version(), ABI_VERSION))
_lib.nsv_strerror.restype = ctypes.c_char_p
_lib.nsv_strerror.argtypes = [_i32]
_lib.nsv_plan_split.restype = _i32
_lib.nsv_plan_split.argtypes = [_SP, _i32, _PP]
_lib.nsv_plan_custom.restype = _i32
_lib.nsv_plan_custom.argtypes = [_SP, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _PP]
_lib.nsv_plan_resident_ctas.restype = _i32
_lib.nsv_plan_resident_ctas.argtypes = [_SP, _PP, ctypes.POINTER(ctypes.c_int)]
_lib.nsv_kv_write.restype = _i32
_lib.nsv_kv_write.argtypes = [_SP, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.nsv_paged_decode.restype = _i32
_lib.nsv_paged_decode.argtypes = [_SP, _vp, _vp, _vp, _vp, _vp, _f, _vp, _vp]
_lib.nsv_paged_decode_ws.restype = _i32
_lib.nsv_paged_decode_ws.argtypes = [_SP, _PP, _vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _sz, _vp]
_lib.nsv_decode_step.restype = _i32
_lib.nsv_decode_step.argtypes = [_SP, _PP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f, _vp,
                                 _vp, _sz, _vp]
_lib.nsv_paged_decode_slots.restype = _i32
_lib.nsv_paged_decode_slots.argtypes = [_SP, _PP, _vp, _vp, _vp, _vp, ctypes.c_int64,
                                        ctypes.c_int64, _vp, _f, _vp, _vp, _sz, _vp]
_lib.nsv_paged_decode_noalloc.restype = _i32
_lib.nsv_paged_decode_noalloc.argtypes = [_SP, _vp, _vp, _vp, _vp, _vp, _f, _vp, _vp]
_lib.nsv_device_status.restype = _i32
_lib.nsv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(ctypes.c_uint64), _i32]
_lib.nsv_status_async.restype = _i32
_lib.nsv_status_async.argtypes = [_vp, _i32, _vp]
_lib.nsv_selftest_bounded_wait.restype = _i32
_lib.nsv_selftest_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_uint64), _vp]


class NsvError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, ERRORS.get(code, code),
                                          _lib.nsv_strerror(code).decode()))


def _check(rc, where):
    if rc != 0:
        raise NsvError(rc, where)


def lib_path():
    return LIB_PATH


def abi_version():
    return _lib.nsv_abi_version()


def strerror(code):
    return _lib.nsv_strerror(code).decode()


def make_shape(rows, num_heads, num_kv_heads, head_dim, max_blocks, num_blocks, dtype,
               block_size=16, query_len=1):
    return Shape(rows, num_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks,
                 dtype, query_len)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("nsv tensors must be float32 or bfloat16, got %s" % t.dtype)


def _ptr(t, what):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    return t.data_ptr()


def shape_of(q, k_pool, block_tables):
    """nsv_shape from the read's tensors (q is [R, H, D] or [R, NQ, H, D])."""
    if q.dim() == 4:
        R, NQ, H, D = q.shape
    else:
        (R, H, D), NQ = q.shape, 1
    NB1, Hkv, B, D2 = k_pool.shape
    if D2 != D:
        raise ValueError("q head_dim %d != pool head_dim %d" % (D, D2))
    if block_tables.shape[0] != R:
        raise ValueError("block_tables rows %d != q rows %d" % (block_tables.shape[0], R))
    if q.dtype != k_pool.dtype:
        raise ValueError("q and the pool must share one dtype")
    return make_shape(R, H, Hkv, D, block_tables.shape[1], NB1 - 1, _dtype_code(k_pool), B,
                      query_len=NQ)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def plan_split(shape, num_sms=0):
    p = Plan()
    _check(_lib.nsv_plan_split(ctypes.byref(shape), int(num_sms), ctypes.byref(p)),
           "nsv_plan_split")
    return p


def plan_custom(shape, num_sms=0, kv_heads_per_cta=0, stages=0, ctas_per_sm=0, grid=0,
                vectors_per_warp=0, consumer=CONSUMER_AUTO, blocks_per_stage=0):
    p = Plan()
    _check(_lib.nsv_plan_custom(ctypes.byref(shape), int(num_sms), int(kv_heads_per_cta),
                                int(stages), int(ctas_per_sm), int(grid), int(vectors_per_warp),
                                int(consumer), int(blocks_per_stage), ctypes.byref(p)),
           "nsv_plan_custom")
    return p


def plan_resident_ctas(shape, plan):
    """CTAs of the plan's kernel that one SM of the current device holds."""
    n = ctypes.c_int(0)
    _check(_lib.nsv_plan_resident_ctas(ctypes.byref(shape), ctypes.byref(plan), ctypes.byref(n)),
           "nsv_plan_resident_ctas")
    return n.value


def workspace_for(plan, device=None):
    """A caller-owned workspace tensor for `plan` (None when it needs none)."""
    import torch
    if plan.workspace_bytes == 0:
        return None
    return torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=device or "cuda")


def kv_write(k_new, v_new, write_slots, k_pool, v_pool, stream=None):
    if k_new.dim() == 4:
        k_new = k_new.reshape(-1, k_new.shape[2], k_new.shape[3])
        v_new = v_new.reshape(-1, v_new.shape[2], v_new.shape[3])
        write_slots = write_slots.reshape(-1)
    R, Hkv, D = k_new.shape
    NB1, Hkv2, B, D2 = k_pool.shape
    if (Hkv, D) != (Hkv2, D2) or k_new.dtype != k_pool.dtype or v_new.dtype != k_pool.dtype:
        raise ValueError("k_new/v_new do not match the pool")
    shape = make_shape(R, Hkv2, Hkv2, D2, 1, NB1 - 1, _dtype_code(k_pool), B)
    _check(_lib.nsv_kv_write(ctypes.byref(shape), _ptr(k_new, "k_new"), _ptr(v_new, "v_new"),
                             _ptr(write_slots, "write_slots"), _ptr(k_pool, "k_pool"),
                             _ptr(v_pool, "v_pool"), _stream(stream)), "nsv_kv_write")


def paged_decode(q, k_pool, v_pool, block_tables, context_lens, scale, out, stream=None):
    """Decode read with the default plan and the library-owned workspace."""
    shape = shape_of(q, k_pool, block_tables)
    _check(_lib.nsv_paged_decode(ctypes.byref(shape), _ptr(q, "q"), _ptr(k_pool, "k_pool"),
                                 _ptr(v_pool, "v_pool"), _ptr(block_tables, "block_tables"),
                                 _ptr(context_lens, "context_lens"), float(scale),
                                 _ptr(out, "out"), _stream(stream)), "nsv_paged_decode")
    return out


def paged_decode_noalloc(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                         stream=None):
    """Decode read that allocates no device memory (scratch from the library's
    fixed buffer; see nsv_paged_decode_noalloc in nsv.h for the size limit)."""
    shape = shape_of(q, k_pool, block_tables)
    _check(_lib.nsv_paged_decode_noalloc(ctypes.byref(shape), _ptr(q, "q"),
                                         _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"),
                                         _ptr(block_tables, "block_tables"),
                                         _ptr(context_lens, "context_lens"), float(scale),
                                         _ptr(out, "out"), _stream(stream)),
           "nsv_paged_decode_noalloc")
    return out


def paged_decode_ws(q, k_pool, v_pool, block_tables, context_lens, scale, out, workspace=None,
                    plan=None, stream=None):
    """Decode read with an explicit plan (None: default) and caller workspace."""
    shape = shape_of(q, k_pool, block_tables)
    ws_ptr = _ptr(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.nsv_paged_decode_ws(ctypes.byref(shape), ctypes.byref(plan) if plan else None,
                                    _ptr(q, "q"), _ptr(k_pool, "k_pool"), _ptr(v_pool, "v_pool"),
                                    _ptr(block_tables, "block_tables"),
                                    _ptr(context_lens, "context_lens"), float(scale),
                                    _ptr(out, "out"), ws_ptr, ws_bytes, _stream(stream)),
           "nsv_paged_decode_ws")
    return out


def paged_decode_slots(q, k_pool, v_pool, slot_table, context_lens, scale, out, workspace=None,
                       plan=None, max_blocks=None, stream=None):
    """Decode read through a per-token slot table.

    slot_table is an int64 [rows, width] tensor whose rows may be strided (a
    window of a wider table, as slots[:rows, :width] of a persistent buffer);
    its last dimension must be contiguous.  max_blocks defaults to
    cdiv(width, 16) and only sizes the plan.
    """
    import torch
    if slot_table.dtype != torch.int64 or slot_table.dim() != 2 or \
            (slot_table.shape[1] > 1 and slot_table.stride(1) != 1):
        raise ValueError("slot_table must be an int64 [rows, width] tensor with unit column stride")
    if not slot_table.is_cuda:
        raise ValueError("slot_table must be a CUDA tensor")
    rows, width = slot_table.shape
    mb = max_blocks or (width + 15) // 16
    if q.dim() == 4:
        R, NQ, H, D = q.shape
    else:
        (R, H, D), NQ = q.shape, 1
    NB1, Hkv, B, _ = k_pool.shape
    shape = make_shape(R, H, Hkv, D, mb, NB1 - 1, _dtype_code(k_pool), B, query_len=NQ)
    ws_ptr = _ptr(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.nsv_paged_decode_slots(ctypes.byref(shape), ctypes.byref(plan) if plan else None,
                                       _ptr(q, "q"), _ptr(k_pool, "k_pool"),
                                       _ptr(v_pool, "v_pool"), slot_table.data_ptr(), int(width),
                                       int(slot_table.stride(0)),
                                       _ptr(context_lens, "context_lens"), float(scale),
                                       _ptr(out, "out"), ws_ptr, ws_bytes, _stream(stream)),
           "nsv_paged_decode_slots")
    return out


def decode_step(q, k_new, v_new, write_slots, k_pool, v_pool, block_tables, context_lens, scale,
                out, workspace=None, plan=None, stream=None):
    """Append then read, on one stream (workspace None: the library's)."""
    shape = shape_of(q, k_pool, block_tables)
    ws_ptr = _ptr(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.nsv_decode_step(ctypes.byref(shape), ctypes.byref(plan) if plan else None,
                                _ptr(q, "q"), _ptr(k_new, "k_new"), _ptr(v_new, "v_new"),
                                _ptr(write_slots, "write_slots"), _ptr(k_pool, "k_pool"),
                                _ptr(v_pool, "v_pool"), _ptr(block_tables, "block_tables"),
                                _ptr(context_lens, "context_lens"), float(scale),
                                _ptr(out, "out"), ws_ptr, ws_bytes, _stream(stream)),
           "nsv_decode_step")
    return out


def selftest_bounded_wait(limit_ns, stream=None):
    """Run the decode kernel's bounded wait on a barrier nothing completes;
    returns (gave_up, waited_ns).  Synchronises the stream."""
    gave_up = ctypes.c_int(0)
    waited = ctypes.c_uint64(0)
    _check(_lib.nsv_selftest_bounded_wait(int(limit_ns), ctypes.byref(gave_up),
                                          ctypes.byref(waited), _stream(stream)),
           "nsv_selftest_bounded_wait")
    return gave_up.value, waited.value


def status_async(dst, clear=True, stream=None):
    """Enqueue a copy of the device status word into `dst` (a uint32/int32
    tensor of at least one element, on the device or in pinned host memory)
    and, with `clear`, zero the word, both on `stream`; no synchronisation.
    Read `dst` once the stream has reached the copy."""
    import torch
    if dst.dtype not in (torch.int32, torch.uint32) or dst.numel() < 1:
        raise ValueError("dst must be an int32 or uint32 tensor of at least one element")
    if not dst.is_cuda and not dst.is_pinned():
        raise ValueError("dst must be device memory or pinned host memory")
    _check(_lib.nsv_status_async(dst.data_ptr(), 1 if clear else 0, _stream(stream)),
           "nsv_status_async")
    return dst


def device_status(clear=True):
    """(status bits, walked (row, block) pairs) of the current device; synchronises."""
    st = ctypes.c_uint32(0)
    w = ctypes.c_uint64(0)
    _check(_lib.nsv_device_status(ctypes.byref(st), ctypes.byref(w), 1 if clear else 0),
           "nsv_device_status")
    return st.value, w.value
