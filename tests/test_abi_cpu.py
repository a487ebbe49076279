"""The C ABI library on a machine without a GPU: it loads, exports every entry
point the header declares, plans work, and rejects bad arguments before it
touches CUDA."""
import ctypes
import os
import re

import pytest
import torch

import grouped_query_decode_gb300 as gq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa_decode.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(gqa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gqa_decode", "gqa_decode_ex", "gqa_decode_workspace_bytes", "gqa_decode_plan",
              "gqa_decode_check_error", "gqa_decode_last_cuda_error", "gqa_decode_strerror",
              "gqa_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(gq.load()._name)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_covers_every_code():
    for code in range(0, -8, -1):
        assert gq.strerror(code) != "unknown status"
    assert gq.strerror(12345) == "unknown status"


def test_plan_shapes():
    # Llama-3-8B-shaped layer: 16 x 8 units x 64 tiles over 152 SMs.
    p = gq.gqa_decode_plan(16, 1, 32, 8, 128, 4096, 152)
    assert p["ctas"] == 152 and p["tile_tokens"] == 64 and p["row_tiles"] == 1
    assert p["max_tiles"] == 16 * 8 * 64
    # 4 consumer warps, the producer warp, the two page-loader warps (idle
    # unless the cache is paged in pages shorter than a tile), the counter warp.
    assert p["smem_bytes"] <= 227 * 1024 and p["threads"] == 256
    # MQA end: 32 rows -> two 16-row tiles: 8 consumers + producer + 2 loaders + counter.
    p = gq.gqa_decode_plan(64, 1, 32, 1, 128, 8192, 152)
    assert p["row_tiles"] == 2 and p["threads"] == 384
    # A tiny problem gets at least 16 tiles (1024 tokens) per CTA.
    p = gq.gqa_decode_plan(1, 1, 32, 8, 64, 1024, 152)
    assert p["max_tiles"] == 128 and p["ctas"] == 8


def test_plan_min_tiles_override(monkeypatch):
    monkeypatch.setenv("GQA_DECODE_MIN_TILES_PER_CTA", "1")
    assert gq.gqa_decode_plan(1, 1, 32, 8, 64, 1024, 152)["ctas"] == 128


@pytest.mark.parametrize("args,code", [
    ((0, 1, 32, 8, 128, 4096), gq.GQA_ERR_INVALID_ARG),
    ((1, 0, 32, 8, 128, 4096), gq.GQA_ERR_INVALID_ARG),
    ((1, 1, 30, 8, 128, 4096), gq.GQA_ERR_HEAD_RATIO),
    ((1, 1, 32, 8, 96, 4096), gq.GQA_ERR_UNSUPPORTED),
    ((1, 2, 32, 1, 128, 4096), gq.GQA_ERR_UNSUPPORTED),  # R = 64 rows
    ((1, 1, 32, 8, 128, 0), gq.GQA_ERR_INVALID_ARG),
])
def test_plan_rejects(args, code):
    with pytest.raises(gq.GQADecodeError) as e:
        gq.gqa_decode_plan(*args, 152)
    assert e.value.status == code


def _call(lib, ptrs, shape, lse=None):
    q, k, v, lens, out = ptrs
    return lib.gqa_decode(q, k, v, lens, 0.125, out, lse, *shape, None)


def test_argument_checks_need_no_gpu():
    lib = gq.load()
    good = (256, 512, 768, 1024, 1280)
    assert _call(lib, (None, 512, 768, 1024, 1280), (1, 1, 32, 8, 128, 64)) == gq.GQA_ERR_INVALID_ARG
    assert _call(lib, good, (1, 1, 32, 6, 128, 64)) == gq.GQA_ERR_HEAD_RATIO
    assert _call(lib, good, (1, 1, 32, 8, 80, 64)) == gq.GQA_ERR_UNSUPPORTED
    # gqa_decode_ex checks alignment before any CUDA call
    rc = lib.gqa_decode_ex(256, 520, 768, 1024, 0.1, 1280, None, 1, 1, 32, 8, 128, 64, 4096,
                           1 << 20, None)
    assert rc == gq.GQA_ERR_MISALIGNED


def test_prefill_argument_checks_need_no_gpu():
    lib = gq.load()
    good = (256, 512, 768, 1024, 1280)

    def call(ptrs, shape):
        q, k, v, lens, out = ptrs
        return lib.gqa_prefill(q, k, v, lens, 0.125, out, None, *shape, None)

    assert call((None, 512, 768, 1024, 1280), (1, 64, 32, 8, 64, 4096)) == gq.GQA_ERR_INVALID_ARG
    assert call(good, (1, 0, 32, 8, 64, 4096)) == gq.GQA_ERR_INVALID_ARG
    assert lib.gqa_prefill(*good[:4], -0.125, good[4], None, 1, 64, 32, 8, 64, 4096, None) == \
        gq.GQA_ERR_INVALID_ARG
    assert call(good, (1, 64, 32, 6, 64, 4096)) == gq.GQA_ERR_HEAD_RATIO
    assert call(good, (1, 64, 32, 8, 96, 4096)) == gq.GQA_ERR_UNSUPPORTED
    assert call((256, 520, 768, 1024, 1280), (1, 64, 32, 8, 64, 4096)) == gq.GQA_ERR_MISALIGNED
    # 2^31 rows of output would overflow the kernel's 32-bit row numbers
    assert call(good, (1 << 16, 1 << 10, 32, 8, 64, 4096)) == gq.GQA_ERR_UNSUPPORTED


def test_binding_refuses_host_tensors_wrong_dtypes_and_shapes():
    """The Python binding passes raw pointers, so it must refuse what the C
    side cannot see: host tensors (a host pointer handed to a kernel),
    another dtype, or shapes that disagree. All of it before any library call."""
    bf = torch.bfloat16
    q = torch.zeros(1, 1, 32, 128, dtype=bf)
    k = torch.zeros(1, 8, 64, 128, dtype=bf)
    lens = torch.zeros(1, dtype=torch.int32)
    out = torch.zeros_like(q)
    for fn in (gq.gqa_decode, gq.gqa_decode_noalloc, gq.gqa_prefill):
        with pytest.raises(TypeError, match="CUDA tensor"):
            fn(q, k, k, lens, 0.1, out)
        with pytest.raises(TypeError, match="must be torch.bfloat16"):
            fn(q.float(), k, k, lens, 0.1, out)
    with pytest.raises(TypeError, match="CUDA tensor"):
        gq.gqa_decode_ex(q, k, k, lens, 0.1, out, None, torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(TypeError, match="CUDA tensor"):
        gq.gqa_decode_append(q, torch.zeros(1, 1, 8, 128, dtype=bf), torch.zeros(1, 1, 8, 128, dtype=bf),
                             k, k, lens, 0.1, out)
    pages = torch.zeros(4, 8, 16, 128, dtype=bf)
    with pytest.raises(TypeError, match="CUDA tensor"):
        gq.gqa_decode_paged(q, pages, pages, torch.zeros(1, 4, dtype=torch.int32), lens, 0.1, out)
    codes = torch.zeros(1, 8, 64, 128, dtype=torch.uint8)
    sc = torch.ones(1, 8, 1)
    with pytest.raises(TypeError, match="CUDA tensor"):
        gq.gqa_decode_fp8(q, codes, codes, sc, sc, lens, 0.1, out)
