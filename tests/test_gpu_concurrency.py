"""Concurrent callers: each stream gets its own library workspace, so steps
enqueued on different streams -- from one host thread or from several --
may overlap on the GPU without their partial slots or arrival counters
mixing. Plans split units over many CTAs so that every step uses them."""
import math
import threading

import numpy as np
import pytest
import torch

import grouped_query_decode_gb300 as gq
import oracle
from gpu_helpers import bf16_to_f64, compare, make_inputs, min_tiles, to_device_bf16

pytestmark = pytest.mark.gpu

D, TMAX = 128, 1200


def _case(seed, H, G, sq, lens):
    B = len(lens)
    q, k, v, lens = make_inputs(B, sq, H, G, D, TMAX, lens, seed=seed)
    dev = dict(q=to_device_bf16(q), k=to_device_bf16(k), v=to_device_bf16(v), l=torch.from_numpy(lens).cuda(),
               out=torch.empty(B, sq, H, D, dtype=torch.bfloat16, device="cuda"),
               lse=torch.empty(B, sq, H, dtype=torch.float32, device="cuda"))
    ref = oracle.gqa_decode_f64(q, k, v, lens, 1 / math.sqrt(D), threads=8)
    return dev, ref


def _check(dev, ref, what):
    compare(bf16_to_f64(dev["out"]), dev["lse"].cpu().numpy().astype(np.float64), ref[0], ref[1], what=what)


def test_two_streams_interleaved():
    cases = [_case(2301, 32, 8, 1, [1200, 700, 77]), _case(2302, 64, 8, 4, [900, 1200, 5]),
             _case(2303, 32, 1, 1, [1100, 300]), _case(2304, 16, 4, 2, [1200, 1199, 640])]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    scale = 1 / math.sqrt(D)
    with min_tiles(1):
        for rep in range(3):
            for i, (dev, _) in enumerate(cases):
                with torch.cuda.stream(streams[i % 2]):
                    gq.gqa_decode(dev["q"], dev["k"], dev["v"], dev["l"], scale, dev["out"], dev["lse"])
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    for i, (dev, ref) in enumerate(cases):
        _check(dev, ref, f"stream {i % 2} case {i}")


def test_host_threads_each_with_a_stream():
    cases = [_case(2401 + i, 32 if i % 2 else 64, 8, 1 if i % 2 else 4, [1200, 650, 33]) for i in range(4)]
    scale = 1 / math.sqrt(D)
    errors = []

    def worker(i):
        try:
            dev, _ = cases[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    gq.gqa_decode(dev["q"], dev["k"], dev["v"], dev["l"], scale, dev["out"], dev["lse"], stream=s)
            s.synchronize()
        except Exception as e:   # reported on the main thread
            errors.append(e)

    with min_tiles(1):
        threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    assert gq.gqa_decode_check_error() == gq.GQA_OK
    for i, (dev, ref) in enumerate(cases):
        _check(dev, ref, f"thread {i}")
