"""Shared helpers of the GPU parity tests: move generator output to the device,
call the CUDA path through the C ABI with guard canaries around the outputs,
and compare with the oracle within the stated tolerances."""
from __future__ import annotations

import contextlib
import os

import numpy as np
import torch

import grouped_query_decode_gb300 as gq
import synthetic as syn

# Tolerances of the parity bar: max-abs error 1e-2 on the bf16 output and 1e-3
# on the fp32 natural-log LSE. The output bar adds bf16's own rounding: the
# format keeps 8 significant bits, so rounding alone moves a value by up to
# 2^-8 |x| (1/64 for |x| in [4, 8), which short sequences with a sharp softmax
# reach). On the decode workloads |out| stays below ~0.1 and the bar is
# 1e-2 + <4e-4.
OUT_ATOL = 1e-2
OUT_RTOL_BF16 = 2.0 ** -8
LSE_ATOL = 1e-3

# Not a gate: the max-abs error over the RMS of the reference output, which
# says how close the result is where |out| is small (about 1/sqrt(T) for
# N(0,1) inputs, so that 1e-2 is a loose bar on long contexts). Tests that
# compute it add a line here; conftest prints them in the terminal summary.
QUALITY: list[str] = []


def note_quality(what, err, ref_out):
    ref = np.asarray(ref_out, dtype=np.float64)
    ref = ref[np.isfinite(ref)]
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    rel = err / rms if rms > 0 else float("nan")
    QUALITY.append(f"{what}: max-abs {err:.2e}, RMS of out {rms:.2e}, ratio {rel:.2e}")
    return rel


_PAD = 64          # guard elements on each side of an output (keeps 16 B alignment)
_CANARY_BF16 = 0x7F7F
_CANARY_F32 = np.float32(-1.2345e29)


def to_device_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


@contextlib.contextmanager
def min_tiles(n):
    old = os.environ.get("GQA_DECODE_MIN_TILES_PER_CTA")
    if n is None:
        os.environ.pop("GQA_DECODE_MIN_TILES_PER_CTA", None)
    else:
        os.environ["GQA_DECODE_MIN_TILES_PER_CTA"] = str(n)
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("GQA_DECODE_MIN_TILES_PER_CTA", None)
        else:
            os.environ["GQA_DECODE_MIN_TILES_PER_CTA"] = old


@contextlib.contextmanager
def env(**kv):
    """Sets (or, with None, unsets) environment variables for the block."""
    old = {k: os.environ.get(k) for k in kv}
    for k, v in kv.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = str(v)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_gpu(q, k, v, lens, scale, with_lse=True, device_inputs=None, entry=None):
    """Runs gqa_decode (or `entry`, a binding with its signature) on the device. Returns (out float64 [B,sq,H,D], lse
    float64 [B,sq,H] or None). Checks that the guard words around out and lse
    are untouched and that no device-side wait expired."""
    if device_inputs is None:
        dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
        dl = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    else:
        dq, dk, dv, dl = device_inputs
    B, sq, H, D = dq.shape
    n = B * sq * H * D
    out_buf = torch.full((n + 2 * _PAD,), 0, dtype=torch.int16, device="cuda")
    out_buf.fill_(np.int16(np.uint16(_CANARY_BF16).view(np.int16)))
    out = out_buf[_PAD:_PAD + n].view(torch.bfloat16).view(B, sq, H, D)
    lse = None
    if with_lse:
        m = B * sq * H
        lse_buf = torch.full((m + 2 * _PAD,), float(_CANARY_F32), dtype=torch.float32, device="cuda")
        lse = lse_buf[_PAD:_PAD + m].view(B, sq, H)
    (entry or gq.gqa_decode)(dq, dk, dv, dl, scale, out, lse)
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    ob = out_buf.cpu().numpy().view(np.uint16)
    assert np.all(ob[:_PAD] == _CANARY_BF16) and np.all(ob[_PAD + n:] == _CANARY_BF16), "out guard"
    lse_np = None
    if with_lse:
        lb = lse_buf.cpu().numpy()
        m = B * sq * H
        assert np.all(lb[:_PAD] == _CANARY_F32) and np.all(lb[_PAD + m:] == _CANARY_F32), "lse guard"
        lse_np = lb[_PAD:_PAD + m].astype(np.float64).reshape(B, sq, H)
    return bf16_to_f64(out), lse_np


def compare(out, lse, ref_out, ref_lse, rows=None, what=""):
    """Max-abs bars on out and lse; rows with no visible key must be exactly
    out = 0 and lse = -inf on both sides."""
    if rows is not None:
        out, ref_out = out.reshape(-1, out.shape[-1])[rows], ref_out.reshape(-1, out.shape[-1])[rows]
        lse, ref_lse = lse.reshape(-1)[rows], ref_lse.reshape(-1)[rows]
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    diff = np.abs(out - ref_out)
    excess = diff - (OUT_ATOL + OUT_RTOL_BF16 * np.abs(ref_out))
    err = diff.max() if out.size else 0.0
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf lse rows differ"
    lerr = np.abs(lse[~empty] - ref_lse[~empty]).max() if (~empty).any() else 0.0
    assert (excess <= 0).all(), (f"{what}: out error {diff.flat[excess.argmax()]:.3e} at "
                                 f"|ref| {np.abs(ref_out).flat[excess.argmax()]:.3e} above "
                                 f"{OUT_ATOL} + 2^-8 |ref|")
    assert lerr <= LSE_ATOL, f"{what}: lse max-abs error {lerr:.3e} > {LSE_ATOL}"
    if empty.any():
        assert np.all(out.reshape(-1, out.shape[-1])[empty.reshape(-1)] == 0), f"{what}: empty rows"
    return float(err), float(lerr)


def make_inputs(B, sq, H, G, D, Tmax, lens, seed, tail=syn.BF16_NAN):
    lens = np.asarray(lens, dtype=np.int32)
    q = syn.normal_bf16(seed, syn.STREAM_Q, (B, sq, H, D))
    k = syn.fill_cache(seed, syn.STREAM_K, B, G, Tmax, D, lens, tail)
    v = syn.fill_cache(seed, syn.STREAM_V, B, G, Tmax, D, lens, tail)
    return q, k, v, lens
