"""GPU parity of the FP8 quantisation at e4m3 rounding boundaries.

The dispatch kernel converts an approximate quotient x * (1 / scale) to e4m3
wherever that cannot change the byte, and the IEEE quotient x / scale where
it could: within a few fp32 ulps of a midpoint between two e4m3 codes, or in
the e4m3 subnormal range.  These inputs put quotients exactly on midpoints
(scales that are powers of two, so x / scale is exact) and within a few ulps
of them (scale and element pairs found by search over BF16 values), plus
elements in the subnormal range.  Every byte and scale must match the
oracle, which divides in IEEE fp32.
"""
import numpy as np
import pytest
import torch

from oracle import ep_oracle as O
from tests import ep_harness as HN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def _bf16_values():
    """Every positive finite BF16 value, as float32."""
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    return (bits << 16).view(np.float32)


def _midpoint_distance(q):
    """Distance in ulps of q's low 20 mantissa bits from an e4m3 midpoint."""
    b = np.abs(q).view(np.uint32) & 0x7FFFFFFF
    return np.abs((b & 0xFFFFF).astype(np.int64) - 0x80000)


def _blocks(rng):
    vals = _bf16_values()
    blocks = []
    # quotients exactly on midpoints: scale 2^k, elements = midpoints * 2^k
    mids = np.array([(1 + (2 * m + 1) / 16) * 2.0 ** e for e in range(-6, 9) for m in range(8)
                     if (1 + (2 * m + 1) / 16) * 2.0 ** e <= 448], dtype=np.float64)
    for k in (-9, -3, 0, 3):
        amax = 448.0 * 2.0 ** k
        x = mids * 2.0 ** k
        for c in range(0, len(x), 127):
            blk = np.concatenate([[amax], x[c:c + 127]])
            blocks.append(blk)
    # scale and element pairs whose IEEE quotient lies within a few ulps of
    # a midpoint (or in the e4m3 subnormal range): search over BF16 amax
    cand = vals[(vals > 1e-3) & (vals < 1e3)]
    amaxes = rng.choice(cand, size=600, replace=False)
    for amax in amaxes:
        s = np.float32(amax) / np.float32(448.0)
        x = vals[(vals > 0) & (vals <= amax)]
        q = (x / s).astype(np.float32)
        d = _midpoint_distance(q)
        near = x[(d <= 24) & (q >= 2.0 ** -6)]
        sub = x[(q < 2.0 ** -6) & (q > 2.0 ** -12)]
        pick = list(near[:100])
        if sub.size:
            pick += list(rng.choice(sub, size=min(8, sub.size), replace=False))
        if near.size:
            blocks.append(np.concatenate([[amax], pick]))
    out = []
    for blk in blocks:
        full = np.zeros(128, dtype=np.float64)
        full[:len(blk)] = blk
        sign = np.where(rng.random(128) < 0.5, -1.0, 1.0)
        sign[0] = 1.0
        out.append(full * sign)
    return np.array(out, dtype=np.float32)


@pytest.mark.parametrize("col_major", [False, True])
def test_fp8_quantisation_at_rounding_boundaries(ep, col_major):
    rng = np.random.default_rng(17)
    blocks = _blocks(rng)
    assert len(blocks) >= 40
    nb = 8
    T = -(-len(blocks) // nb)
    xf = np.zeros((T * nb, 128), dtype=np.float32)
    xf[:len(blocks)] = blocks
    x = torch.from_numpy(xf.reshape(T, nb * 128)).to(torch.bfloat16)
    # every element survives the BF16 cast unchanged (they are BF16 values)
    assert np.array_equal(x.float().numpy().reshape(-1, 128)[:len(blocks)], blocks)
    H = nb * 128
    K, E, R = 2, 8, 2
    idx = torch.tensor([[t % E, (t + 3) % E] for t in range(T)], dtype=torch.int64)
    w = torch.full((T, K), 0.5)
    cfg = ep.make_config(T, K, E, R, H, T, 4, True, True, True, True, col_major)
    dev = torch.device("cuda")
    h = ep.ep_layout(cfg, idx.to(dev))
    lay = HN.oracle_layout(cfg, idx.numpy())
    HN.check_layout(h, lay)
    out = ep.alloc_recv(h, with_weights=True)
    ep.ep_dispatch(h, x.to(dev), w.to(dev), **out)
    d_or = O.dispatch(lay, HN.bits16(x), w.numpy(), True, col_major, True)
    HN.check_dispatch(h, lay, d_or, out, True, col_major)
    h.free()
