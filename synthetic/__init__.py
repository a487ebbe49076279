"""Seeded synthetic inputs shared by the oracle's tests, the GPU parity tests and
the bench. Holds no attention arithmetic: it only draws numbers (see gen.c for
the counter-based SplitMix64 + Box-Muller definition) and lays them out as the
decode workloads' tensors.

Tensors are returned as numpy arrays of bf16 *bit patterns* (uint16), so that
the oracle (which converts bf16 bits to double exactly) and the GPU path (which
reinterprets the same bits as torch.bfloat16) read identical values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import CONFIGS, PREFILL_CONFIGS, DecodeConfig, config_by_name  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()

# Stream ids: one independent counter stream per tensor.
STREAM_Q, STREAM_K, STREAM_V, STREAM_LENS = 1, 2, 3, 4
BF16_NAN = 0x7FC0
BF16_ZERO = 0x0000


def build(force: bool = False) -> str:
    """Compiles gen.c into libsynth.so beside it (plain gcc, no GPU needed)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
            vp = ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, vp]
            lib.synth_normal_bf16.restype = None
            lib.synth_uniform_int.argtypes = [u64, u64, u64, u64, i64, i64, vp]
            lib.synth_uniform_int.restype = None
            lib.synth_fill_cache.argtypes = [
                u64, u64, i32, i32, i32, i32, vp, ctypes.c_uint16, i32, i32, vp
            ]
            lib.synth_fill_cache.restype = None
            _lib = lib
    return _lib


def normal_bf16(seed: int, stream: int, shape, first: int = 0) -> np.ndarray:
    """N(0,1) draws rounded to bf16, as uint16 bits; element j (flat, C order)
    is the draw at counter index first + j."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, stream, first, n, out.ctypes.data)
    return out.reshape(shape)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, first: int = 0) -> np.ndarray:
    """Integers uniform in [lo, hi], both ends inclusive."""
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_uniform_int(seed, stream, first, n, lo, hi, out.ctypes.data)
    return out


def _threads(threads):
    if threads is None:
        threads = os.cpu_count() or 1
    return max(1, int(threads))


def fill_cache(seed: int, stream: int, B: int, G: int, Tmax: int, D: int,
               seq_lens: np.ndarray, tail_bits: int, out: np.ndarray | None = None,
               threads: int | None = None) -> np.ndarray:
    """A [B, G, Tmax, D] cache: element (b,g,t,d) with t < seq_lens[b] is the draw
    at flat index ((b*G+g)*Tmax+t)*D+d; the tail t >= seq_lens[b] holds tail_bits
    (NaN for parity runs, so that any read past the valid length poisons the
    result; zero for timed runs). `out` may be any C-contiguous uint16 buffer of
    that size (e.g. a pinned host tensor's numpy view)."""
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert lens.shape == (B,)
    if out is None:
        out = np.empty((B, G, Tmax, D), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"] and out.size == B * G * Tmax * D
    lib = _load()
    nt = min(_threads(threads), B)
    bounds = [(B * i) // nt for i in range(nt + 1)]

    def work(i):
        lib.synth_fill_cache(seed, stream, B, G, Tmax, D, lens.ctypes.data, tail_bits,
                             bounds[i], bounds[i + 1], out.ctypes.data)

    if nt == 1:
        work(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, range(nt)))
    return out.reshape(B, G, Tmax, D)


def cache_slice(seed: int, stream: int, G: int, Tmax: int, D: int, b: int, g: int,
                T: int) -> np.ndarray:
    """Rows [0, T) of unit (b, g) of a cache made by fill_cache with the same
    seed/stream/G/Tmax/D, regenerated on its own: [T, D] uint16."""
    first = ((b * G + g) * Tmax) * D
    return normal_bf16(seed, stream, (T, D), first=first)


def seq_lens_for(cfg: DecodeConfig) -> np.ndarray:
    """Per-sequence valid lengths (including the sq new tokens) of a workload."""
    if cfg.t_lo == cfg.t_hi:
        return np.full(cfg.B, cfg.t_hi, dtype=np.int32)
    return uniform_int(cfg.seed, STREAM_LENS, cfg.B, cfg.t_lo, cfg.t_hi)


def make_inputs(cfg: DecodeConfig, tail_bits: int = BF16_NAN, threads: int | None = None,
                seq_lens: np.ndarray | None = None):
    """q [B,sq,H,D], k/v caches [B,G,Tmax,D] (bf16 bits) and seq_lens [B] int32."""
    lens = seq_lens_for(cfg) if seq_lens is None else np.asarray(seq_lens, dtype=np.int32)
    q = normal_bf16(cfg.seed, STREAM_Q, (cfg.B, cfg.sq, cfg.H, cfg.D))
    k = fill_cache(cfg.seed, STREAM_K, cfg.B, cfg.G, cfg.Tmax, cfg.D, lens, tail_bits,
                   threads=threads)
    v = fill_cache(cfg.seed, STREAM_V, cfg.B, cfg.G, cfg.Tmax, cfg.D, lens, tail_bits,
                   threads=threads)
    return q, k, v, lens


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round-to-nearest-even (NaN kept as a quiet NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7F800000) == 0x7F800000
    nan &= (u & 0x007FFFFF) != 0
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = BF16_NAN
    return r


def paginate(k: np.ndarray, v: np.ndarray, seq_lens: np.ndarray, page_size: int, seed: int,
             spare_pages: int = 3, fill_bits: int = BF16_NAN):
    """Lays contiguous caches [B, G, Tmax, D] out as pages [num_pages, G,
    page_size, D] in a seeded random physical order. Every page that holds a
    token before a sequence's length is placed; the spare pages and the
    unused block-table entries point at NaN-filled pages, whose contents a
    step must never let into its result. Returns (k_pages, v_pages,
    block_table [B, max_pages] int32)."""
    B, G, Tmax, D = k.shape
    max_pages = -(-Tmax // page_size)
    lens = np.clip(np.asarray(seq_lens, dtype=np.int64), 0, Tmax)
    need = [int(-(-int(t) // page_size)) for t in lens]
    num_pages = sum(need) + spare_pages
    order = np.argsort(uniform_int(seed, 21, num_pages, 0, 2**31 - 1), kind="stable")
    kp = np.full((num_pages, G, page_size, D), fill_bits, dtype=np.uint16)
    vp = np.full((num_pages, G, page_size, D), fill_bits, dtype=np.uint16)
    table = np.empty((B, max_pages), dtype=np.int32)
    spare = [int(x) for x in order[sum(need):]] or [0]
    nxt = 0
    for b in range(B):
        for j in range(max_pages):
            if j < need[b]:
                phys = int(order[nxt])
                nxt += 1
                rows = slice(j * page_size, min((j + 1) * page_size, Tmax))
                n = rows.stop - rows.start
                kp[phys, :, :n] = k[b, :, rows]
                vp[phys, :, :n] = v[b, :, rows]
                table[b, j] = phys
            else:
                table[b, j] = spare[(b + j) % len(spare)]
    return kp, vp, table


E4M3_NAN = 0x7F


def fp8_cache(bits: np.ndarray, seq_lens: np.ndarray, tail_code: int = E4M3_NAN):
    """An fp8 (OCP E4M3) version of a bf16 cache [B, G, Tmax, D]: one fp32
    scale per 64-token block of each (sequence, KV head), amax / 448 over the
    block's valid rows (1 for a block with none), and codes = the e4m3
    rounding (torch's float8_e4m3fn cast, round to nearest even) of
    value / scale. Rows at or past a sequence's length get tail_code (NaN by
    default). Returns (codes uint8 [B, G, Tmax, D], scales float32
    [B, G, ceil(Tmax / 64)])."""
    import torch
    B, G, Tmax, D = bits.shape
    nt = -(-Tmax // 64)
    x = torch.from_numpy(bf16_bits_to_f32(bits).reshape(B, G, Tmax, D))
    lens = np.clip(np.asarray(seq_lens, dtype=np.int64), 0, Tmax)
    valid = torch.arange(Tmax)[None, :] < torch.from_numpy(lens)[:, None]          # [B, Tmax]
    xv = torch.where(valid[:, None, :, None], x, torch.zeros(()))
    pad = nt * 64 - Tmax
    amax = torch.nn.functional.pad(xv.abs(), (0, 0, 0, pad)).reshape(B, G, nt, 64 * D).amax(-1)
    scales = torch.where(amax > 0, amax / 448.0, torch.ones(()))                     # [B, G, nt]
    per_row = scales.repeat_interleave(64, dim=2)[:, :, :Tmax, None]
    codes = (x / per_row).to(torch.float8_e4m3fn).view(torch.uint8)
    codes = torch.where(valid[:, None, :, None], codes, torch.full((), tail_code, dtype=torch.uint8))
    return codes.numpy().copy(), scales.numpy().astype(np.float32).copy()
