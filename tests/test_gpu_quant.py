"""GPU MXFP8 quantisation vs the oracle, bit-exact (E4M3 bytes and E8M0 scales)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_build_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mok():
    from mixture_experts_layer_build_gb300 import mok as m
    return m


def _rand_bits(rng, rows, cols, lo=-30, hi=30):
    v = rng.standard_normal((rows, cols)).astype(np.float32) * (2.0 ** rng.integers(lo, hi, size=(rows, 1)))
    return inputs.bits(torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16))


@pytest.mark.parametrize("rows,cols,seed", [(1, 32, 0), (64, 256, 1), (257, 96, 2), (33, 7168, 3)])
def test_quantize_bit_exact(mok, rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = _rand_bits(rng, rows, cols)
    q, s = mok.mok_mxfp8_quantize(inputs.from_bits(x).cuda())
    rq, rs = oracle.mxfp8_quantize(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantize_every_bf16_pattern(mok):
    # all 65536 bf16 patterns, in blocks whose amax spans the whole exponent range
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    rng = np.random.default_rng(4)
    x = rng.permutation(allbits).reshape(-1, 64)
    q, s = mok.mok_mxfp8_quantize(inputs.from_bits(x).cuda())
    rq, rs = oracle.mxfp8_quantize(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)
    # sorted blocks: magnitudes close to each other, exercising every rounding position
    xs = np.sort(allbits[(allbits & 0x7F80) != 0x7F80]).reshape(-1, 32)
    q, s = mok.mok_mxfp8_quantize(inputs.from_bits(np.ascontiguousarray(xs)).cuda())
    rq, rs = oracle.mxfp8_quantize(np.ascontiguousarray(xs))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantize_special_blocks(mok):
    x = np.zeros((4, 64), np.uint16)
    x[1, :32] = 0x3F80
    x[1, 32:] = 0x8000
    x[2, 5] = 0x7FC0
    x[2, 40] = 0xFF80
    x[3, :] = 0x0001  # smallest subnormal bf16 everywhere
    q, s = mok.mok_mxfp8_quantize(inputs.from_bits(x).cuda())
    rq, rs = oracle.mxfp8_quantize(x)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantize_weight_sized_sampled_rows(mok):
    # a full per-expert weight of the EP64-shard shape on the GPU; the oracle checks sampled rows
    g = torch.Generator(device="cuda").manual_seed(0)
    w = (torch.randn((2048, 7168), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    q, s = mok.mok_mxfp8_quantize(w)
    rows = np.random.default_rng(0).choice(2048, size=64, replace=False)
    xb = inputs.bits(w[torch.from_numpy(rows).cuda()])
    rq, rs = oracle.mxfp8_quantize(xb)
    assert np.array_equal(q[torch.from_numpy(rows).cuda()].cpu().numpy(), rq)
    assert np.array_equal(s[torch.from_numpy(rows).cuda()].cpu().numpy(), rs)


def test_quantize_rejects_ragged(mok):
    with pytest.raises(mok.MokError):
        mok.mok_mxfp8_quantize(torch.zeros((2, 48), dtype=torch.bfloat16, device="cuda"))
