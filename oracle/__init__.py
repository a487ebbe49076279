"""CPU oracle for grouped-query decode attention (fp64, plain loops in C).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
bench's CPU-baseline / reference arm may import this module; the GPU path never
does, and shares no code with it. See gqa_oracle.c for the definition it
follows ("GQA analysis", section "Grouped broadcast"; bottom-right causal mask
for several new tokens per the mask-handling part of section 7 of "Same GQA,
Different Execution Cost Across Backends").

Every function here is pinned by the `-m "not gpu"` tests in tests/ against
facts that do not come from the oracle itself (the head-mapping table printed
on the first page, repeat_kv / repeat_interleave expansion, PyTorch's own
scaled_dot_product_attention in float64, high-precision brute force, closed
forms); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gqa.so")
_lock = threading.Lock()
_default = None


def compile_oracle(src: str, out_path: str) -> str:
    """Plain gcc build of an oracle source file into a shared library."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"])
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE)
    ):
        compile_oracle(SOURCE, _LIB_PATH)
    return _LIB_PATH


class Oracle:
    """ctypes handle on one build of the oracle (the real one, or a test's
    deliberately broken copy)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        vp, i32, lng = ctypes.c_void_p, ctypes.c_int, ctypes.c_long
        lib.oracle_gqa_decode_f64.argtypes = [vp, vp, vp, vp, ctypes.c_double,
                                              i32, i32, i32, i32, i32, i32, lng, lng, vp, vp]
        lib.oracle_gqa_decode_f64.restype = ctypes.c_int
        if hasattr(lib, "oracle_gqa_decode_kvf64"):
            lib.oracle_gqa_decode_kvf64.argtypes = lib.oracle_gqa_decode_f64.argtypes
            lib.oracle_gqa_decode_kvf64.restype = ctypes.c_int
        self._lib = lib
        self.path = lib_path

    def gqa_decode_kv(self, q, k, v, seq_lens, scale, rows=None, threads: int = 1):
        """As gqa_decode, with k and v given as float64 arrays."""
        return self._run(self._lib.oracle_gqa_decode_kvf64, q,
                         np.ascontiguousarray(k, dtype=np.float64),
                         np.ascontiguousarray(v, dtype=np.float64), seq_lens, scale, rows, threads)

    def gqa_decode(self, q, k, v, seq_lens, scale, rows=None, threads: int = 1):
        """q [B,sq,H,D], k/v [B,G,Tmax,D] as bf16 bit arrays (uint16); seq_lens [B].

        Returns (out [B,sq,H,D] float64, lse [B,sq,H] float64). With `rows`
        = (begin, end) only those flat rows r = (b*sq+s)*H+h are computed; the
        others are left NaN. `threads` splits the rows over host threads (each
        row is still computed by one thread in index order, so the result does
        not depend on the split)."""
        return self._run(self._lib.oracle_gqa_decode_f64, q, np.ascontiguousarray(k, dtype=np.uint16),
                         np.ascontiguousarray(v, dtype=np.uint16), seq_lens, scale, rows, threads)

    def _run(self, fn, q, k, v, seq_lens, scale, rows, threads):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, sq, H, D = q.shape
        Bk, G, Tmax, Dk = k.shape
        if (Bk, Dk) != (B, D) or v.shape != k.shape or lens.shape != (B,):
            raise ValueError("shape mismatch")
        out = np.full((B, sq, H, D), np.nan)
        lse = np.full((B, sq, H), np.nan)
        nrows = B * sq * H
        r0, r1 = (0, nrows) if rows is None else rows
        threads = max(1, min(int(threads), r1 - r0 if r1 > r0 else 1))
        bounds = [r0 + ((r1 - r0) * i) // threads for i in range(threads + 1)]

        def work(i):
            return fn(
                q.ctypes.data, k.ctypes.data, v.ctypes.data, lens.ctypes.data, float(scale),
                B, sq, H, G, D, Tmax, bounds[i], bounds[i + 1], out.ctypes.data, lse.ctypes.data)

        if threads == 1:
            rcs = [work(0)]
        else:
            with ThreadPoolExecutor(threads) as ex:
                rcs = list(ex.map(work, range(threads)))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected the arguments")
        return out, lse


def append_f64(k_cache, v_cache, k_new, v_new, seq_lens):
    """The cache update of "GQA analysis", sections "Projection and RoPE" and
    "Incremental decode" (append(K_cache, K_t); append(V_cache, V_t)): new
    token s of sequence b goes to position T_b - sq + s of every KV head, where
    T_b = seq_lens[b] counts the entries including the new ones; positions
    below 0 are dropped. Returns updated copies; k_new/v_new are [B, sq, G, D]
    bf16 bits, the caches [B, G, Tmax, D]."""
    k = np.array(k_cache, dtype=np.uint16, copy=True)
    v = np.array(v_cache, dtype=np.uint16, copy=True)
    B, G, Tmax, D = k.shape
    sq = k_new.shape[1]
    for b in range(B):
        T = int(seq_lens[b])
        for s in range(sq):
            t = T - sq + s
            if 0 <= t < Tmax:
                k[b, :, t, :] = k_new[b, s]
                v[b, :, t, :] = v_new[b, s]
    return k, v


def gqa_decode_append_f64(q, k_cache, v_cache, k_new, v_new, seq_lens, scale, threads: int = 1):
    """Append the new tokens' K/V (append_f64), then the decode definition over
    the updated caches. Returns (out, lse, k_cache_after, v_cache_after)."""
    k, v = append_f64(k_cache, v_cache, k_new, v_new, seq_lens)
    out, lse = get().gqa_decode(q, k, v, seq_lens, scale, threads=threads)
    return out, lse, k, v


def gather_pages(k_pages, block_table, seq_lens, Tmax):
    """The logical [B, G, Tmax, D] cache behind a paged one (PagedAttention's
    placement, which "GQA analysis" names as orthogonal to GQA): token t of
    sequence b lives in page block_table[b, t // page_size] at row
    t % page_size. Only tokens before seq_lens[b] are gathered; the rest of
    the logical cache is NaN (never read by the definition)."""
    num_pages, G, ps, D = k_pages.shape
    B = block_table.shape[0]
    out = np.full((B, G, Tmax, D), 0x7FC0, dtype=np.uint16)
    for b in range(B):
        for t in range(min(int(seq_lens[b]), Tmax)):
            out[b, :, t, :] = k_pages[int(block_table[b, t // ps]), :, t % ps, :]
    return out


def gqa_decode_paged_f64(q, k_pages, v_pages, block_table, seq_lens, scale, threads: int = 1):
    """The decode definition over the logical caches a paged cache holds."""
    ps = k_pages.shape[2]
    Tmax = block_table.shape[1] * ps
    k = gather_pages(k_pages, block_table, seq_lens, Tmax)
    v = gather_pages(v_pages, block_table, seq_lens, Tmax)
    return get().gqa_decode(q, k, v, seq_lens, scale, threads=threads)


def e4m3_to_f64(codes) -> np.ndarray:
    """OCP FP8 E4M3 codes to their values: sign bit, 4 exponent bits with bias
    7, 3 mantissa bits; exponent 0 is subnormal (m * 2^-9); no infinities, and
    S.1111.111 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def dequantize_fp8(codes, scales) -> np.ndarray:
    """The values of an fp8 cache: [B, G, Tmax, D] codes times the scale of
    their 64-token block (scales [B, G, ceil(Tmax/64)])."""
    B, G, Tmax, D = codes.shape
    per_row = np.repeat(np.asarray(scales, dtype=np.float64), 64, axis=2)[:, :, :Tmax, None]
    return e4m3_to_f64(codes) * per_row


def gqa_decode_fp8_f64(q, k_codes, v_codes, k_scale, v_scale, seq_lens, scale, rows=None,
                       threads: int = 1):
    """The decode definition over the dequantised fp8 caches (KV-cache
    quantisation changes only the element precision, "GQA analysis")."""
    return get().gqa_decode_kv(q, dequantize_fp8(k_codes, k_scale), dequantize_fp8(v_codes, v_scale),
                               seq_lens, scale, rows=rows, threads=threads)


def get() -> Oracle:
    """The oracle built from gqa_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gqa_decode_f64(q, k, v, seq_lens, scale, rows=None, threads: int = 1):
    return get().gqa_decode(q, k, v, seq_lens, scale, rows=rows, threads=threads)
