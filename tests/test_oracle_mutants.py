"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant's pins run in a child process (tests/run_pins_on.py), so that a
mutant which crashes is caught rather than ending the session.

Every mutant is a one-place textual edit of nsv_oracle.c (a dropped term, a
wrong sign, a wrong or transposed index, an off-by-one mask, the wrong
operand), compiled into a temporary library on the CPU.  If some plausible
mistake could slip past every pin, the pins would not be pinning the oracle.
"""

import os
import subprocess
import sys

import pytest

import oracle

MUTANTS = {
    "drop_scale": ("s[t] = scale * acc;", "s[t] = acc;"),
    "mask_off_by_one": ("s[t] = (t < c) ? s[t] : -INFINITY;",
                        "s[t] = (t <= c && t < W) ? s[t] : -INFINITY;"),
    "kv_head_modulo": ("int64_t g = h / group;", "int64_t g = h % Hkv;"),
    "pool_layout_transposed": ("base = ((b * Hkv + g) * B + t % B) * D;",
                               "base = ((b * B + t % B) * Hkv + g) * D;"),
    "token_offset_shifted": ("base = ((b * Hkv + g) * B + t % B) * D;",
                             "base = ((b * Hkv + g) * B + (t + 1) % B) * D;"),
    "slot_offset_shifted": ("base = (((sl / B) * Hkv + g) * B + sl % B) * D;",
                            "base = (((sl / B) * Hkv + g) * B + (sl + 1) % B) * D;"),
    "slot_no_negative_wrap": ("sl += pool_blocks * B; /* wraps, as in Python */",
                              "sl = 0;"),
    "slot_row_stride_ignored": ("int64_t sl = slots[r * stride + t];",
                                "int64_t sl = slots[r * W + t];"),
    "softmax_sign": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "no_normalisation": ("s[t] /= z;", "s[t] /= 1.0;"),
    "pv_uses_keys": ("o[d] += s[t] * Vrect[t * D + d];", "o[d] += s[t] * Krect[t * D + d];"),
    "query_transposed": ("qv[d] = widen(q, dtype, ((r * NQ + jq) * H + h) * D + d);",
                         "qv[d] = widen(q, dtype, ((h * NQ + jq) * R + r) * D + d);"),
    "causal_offset_reversed": ("int64_t c = context_lens[r] - (NQ - 1 - jq);",
                               "int64_t c = context_lens[r] - jq;"),
    "causal_window_ignored": ("int64_t c = context_lens[r] - (NQ - 1 - jq);",
                              "int64_t c = context_lens[r];"),
    "no_negative_wrap": ("b += pool_blocks;", "b = 0;"),
    "kv_write_swaps_k_v": ("memcpy((char *)k_pool + dst, (const char *)k_new + src,",
                           "memcpy((char *)k_pool + dst, (const char *)v_new + src,"),
    "kv_write_offset_dropped": ("int64_t blk = write_slots[r] / B, off = write_slots[r] % B;",
                                "int64_t blk = write_slots[r] / B, off = 0;"),
    "walk_floor_not_ceil": ("n += (context_lens[r] + tile - 1) / tile;",
                            "n += context_lens[r] / tile;"),
    "rect_bytes_fp16": ("return R * H * width * 4;", "return R * H * width * 2;"),
}


RUNNER = os.path.join(os.path.dirname(os.path.abspath(__file__)), "run_pins_on.py")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(oracle.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation site for %s must occur exactly once" % name
    path = os.path.join(str(tmp_path), "mutant_%s.c" % name)
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(str(tmp_path), "libmutant_%s.so" % name))
    # A child process runs the pins: a failing pin exits 1, a crash exits with
    # a signal; both mean the mistake was caught.
    r = subprocess.run([sys.executable, RUNNER, lib], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, "mutant %s passed every pin" % name


def test_runner_passes_the_real_oracle():
    r = subprocess.run([sys.executable, RUNNER, oracle.build()], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
