"""The oracle for the batched paged-attention decode read and the KV append.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only callers.  The product
package never imports this module, and this module imports nothing from the
product package.

The arithmetic lives in ``nsv_oracle.c`` (plain C, fp64), which states what
each function follows on the nanoserve pages.  This file only compiles it
with gcc and marshals numpy arrays to it.

Array conventions (numpy, C-contiguous):
  q, out            [rows, heads, head_dim]
  k_pool, v_pool    [num_blocks + 1, kv_heads, block_size, head_dim]
                    (the last block is the sink block)
  k_new, v_new      [rows, kv_heads, head_dim]
  block_tables      [rows, max_blocks] int32 (padding may be -1)
  context_lens      [rows] int32
  write_slots       [rows] int64
fp32 data is ``np.float32``; bf16 data is ``np.uint16`` holding the raw bf16
bit patterns.
"""

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "nsv_oracle.c")
LIB = os.path.join(_HERE, "liboracle_nsv.so")

F32, BF16 = 0, 1


def compile_source(src_path, out_path):
    """gcc one oracle source file into a shared library."""
    tmp = out_path + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force=False):
    """Compile the oracle into a shared library beside its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_source(SRC, LIB)


class OracleRefusal(ValueError):
    """The oracle refused its inputs (it returns the code it refused with)."""

    def __init__(self, code):
        super().__init__("oracle refused its inputs (code %d)" % code)
        self.code = code


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("oracle data must be float32 or uint16 (bf16 bits), got %s" % arr.dtype)


def _c(arr, dtype):
    out = np.ascontiguousarray(arr, dtype=dtype)
    return out, out.ctypes.data


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_paged_decode.restype = i32
        lib.oracle_paged_decode.argtypes = [i64, i64, i64, i64, i64, i64, i64, i64, i32,
                                            vp, vp, vp, vp, vp, dbl, vp, i64, i32, vp]
        lib.oracle_paged_decode_slots.restype = i32
        lib.oracle_paged_decode_slots.argtypes = [i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                                  i32, vp, vp, vp, vp, vp, dbl, vp, i64, i32,
                                                  vp]
        lib.oracle_kv_write.restype = i32
        lib.oracle_kv_write.argtypes = [i64, i64, i64, i64, i64, i32, vp, vp, vp, vp, vp]
        lib.oracle_walked_tiles.restype = i64
        lib.oracle_walked_tiles.argtypes = [vp, i64, i64]
        lib.oracle_rect_tiles.restype = i64
        lib.oracle_rect_tiles.argtypes = [i64, i64, i64]
        lib.oracle_score_rect_bytes.restype = i64
        lib.oracle_score_rect_bytes.argtypes = [i64, i64, i64]
        lib.oracle_score_tile_bytes.restype = i64
        lib.oracle_score_tile_bytes.argtypes = [i64, i64, i64]
        lib.oracle_max_threads.restype = i32
        lib.oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    def max_threads(self):
        return int(self.lib.oracle_max_threads())

    def paged_decode(self, q, k_pool, v_pool, block_tables, context_lens, scale,
                     rows=None, threads=0):
        """The reference read for the selected rows.

        q is [R, H, D] (one query token per row; returns fp64 [len(rows), H, D])
        or [R, NQ, H, D] (NQ query tokens per row, causal among themselves;
        returns fp64 [len(rows), NQ, H, D]).
        """
        dt = _dtype_code(k_pool)
        if _dtype_code(q) != dt or _dtype_code(v_pool) != dt:
            raise TypeError("q, k_pool and v_pool must share one dtype")
        single = q.ndim == 3
        if single:
            q = q[:, None]
        R, NQ, H, D = q.shape
        NB1, Hkv, B, D2 = k_pool.shape
        if D2 != D or v_pool.shape != k_pool.shape:
            raise ValueError("pool shape does not match q")
        MB = block_tables.shape[1]
        q, qp = _c(q, q.dtype)
        k_pool, kp = _c(k_pool, k_pool.dtype)
        v_pool, vpp = _c(v_pool, v_pool.dtype)
        bt, btp = _c(block_tables, np.int32)
        cl, clp = _c(context_lens, np.int32)
        if rows is None:
            rp, nrows = None, R
        else:
            rows_arr, rp = _c(np.asarray(rows, dtype=np.int64), np.int64)
            nrows = rows_arr.shape[0]
        out = np.zeros((nrows, NQ, H, D), dtype=np.float64)
        rc = self.lib.oracle_paged_decode(R, NQ, H, Hkv, D, B, MB, NB1 - 1, dt, qp, kp, vpp,
                                          btp, clp, float(scale), rp, nrows,
                                          int(threads), out.ctypes.data)
        if rc != 0:
            raise OracleRefusal(rc)
        return out[:, 0] if single else out

    def paged_decode_slots(self, q, k_pool, v_pool, slot_table, width, context_lens, scale,
                           rows=None, threads=0):
        """The read through a per-token slot table [R, stride] (int64; the
        first `width` columns are the rectangle).  Shapes as paged_decode."""
        dt = _dtype_code(k_pool)
        if _dtype_code(q) != dt or _dtype_code(v_pool) != dt:
            raise TypeError("q, k_pool and v_pool must share one dtype")
        single = q.ndim == 3
        if single:
            q = q[:, None]
        R, NQ, H, D = q.shape
        NB1, Hkv, B, D2 = k_pool.shape
        if D2 != D or v_pool.shape != k_pool.shape:
            raise ValueError("pool shape does not match q")
        q, qp = _c(q, q.dtype)
        k_pool, kp = _c(k_pool, k_pool.dtype)
        v_pool, vpp = _c(v_pool, v_pool.dtype)
        st, stp = _c(slot_table, np.int64)
        cl, clp = _c(context_lens, np.int32)
        if rows is None:
            rp, nrows = None, R
        else:
            rows_arr, rp = _c(np.asarray(rows, dtype=np.int64), np.int64)
            nrows = rows_arr.shape[0]
        out = np.zeros((nrows, NQ, H, D), dtype=np.float64)
        rc = self.lib.oracle_paged_decode_slots(R, NQ, H, Hkv, D, B, int(width), st.shape[1],
                                                NB1 - 1, dt, qp, kp, vpp, stp, clp,
                                                float(scale), rp, nrows, int(threads),
                                                out.ctypes.data)
        if rc != 0:
            raise OracleRefusal(rc)
        return out[:, 0] if single else out

    def kv_write(self, k_new, v_new, write_slots, k_pool, v_pool):
        """The KV append, in place on the numpy pools."""
        dt = _dtype_code(k_pool)
        if not (k_pool.flags.c_contiguous and v_pool.flags.c_contiguous):
            raise ValueError("pools must be C-contiguous (they are written in place)")
        R, Hkv, D = k_new.shape
        NB1, Hkv2, B, D2 = k_pool.shape
        if (Hkv2, D2) != (Hkv, D) or v_pool.shape != k_pool.shape:
            raise ValueError("shape mismatch")
        kn, knp = _c(k_new, k_pool.dtype)
        vn, vnp = _c(v_new, k_pool.dtype)
        ws, wsp = _c(write_slots, np.int64)
        rc = self.lib.oracle_kv_write(R, Hkv, D, B, NB1 - 1, dt, knp, vnp, wsp,
                                      k_pool.ctypes.data, v_pool.ctypes.data)
        if rc != 0:
            raise OracleRefusal(rc)

    def walked_tiles(self, context_lens, tile):
        cl, clp = _c(context_lens, np.int32)
        return int(self.lib.oracle_walked_tiles(clp, cl.shape[0], int(tile)))

    def rect_tiles(self, rows, width, tile):
        return int(self.lib.oracle_rect_tiles(int(rows), int(width), int(tile)))

    def score_rect_bytes(self, rows, heads, width):
        return int(self.lib.oracle_score_rect_bytes(int(rows), int(heads), int(width)))

    def score_tile_bytes(self, rows, heads, tile):
        return int(self.lib.oracle_score_tile_bytes(int(rows), int(heads), int(tile)))


_default = None


def default():
    """The oracle built from nsv_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def max_threads():
    return default().max_threads()


def paged_decode(*args, **kwargs):
    return default().paged_decode(*args, **kwargs)


def paged_decode_slots(*args, **kwargs):
    return default().paged_decode_slots(*args, **kwargs)


def kv_write(*args, **kwargs):
    return default().kv_write(*args, **kwargs)


def walked_tiles(context_lens, tile):
    return default().walked_tiles(context_lens, tile)


def rect_tiles(rows, width, tile):
    return default().rect_tiles(rows, width, tile)


def score_rect_bytes(rows, heads, width):
    return default().score_rect_bytes(rows, heads, width)


def score_tile_bytes(rows, heads, tile):
    return default().score_tile_bytes(rows, heads, tile)
