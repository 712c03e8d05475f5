"""GPU parity at wide logical-rank counts, against the oracle.

The DeepEP README's low-latency performance table runs expert parallelism
from 8 up to 256 ranks, and the configuration accepts any rank count that
divides the expert count.  The layout count kernel builds each token's rank
set three ways, by rank count: a 32-bit ballot (R <= 32), a walk over a
64-bit mask (33 <= R <= 64) and, above 64 ranks, a look-back over the
token's earlier slots with is_token_in_rank written byte by byte.  The
cluster kernel (rank layouts of at most 15 chunks) ranks by rank key at any
rank count, with a per-warp rank histogram whose size grows with R.  These
cases run the two wide count branches and the cluster kernel at 48, 64, 128
and 256 ranks through layout, dispatch and combine, in both layouts, with
and without the host count wait, BF16 and FP8 (both scale layouts), with
token counts that span several layout chunks per source rank and a ragged
last chunk, plus one full-size 256-rank decode batch.  Each case states the
layout form it must take.

Layout, metadata and dispatch bytes must match bit for bit; combine within
1 BF16 ulp (and in practice exactly).
"""
import zlib

import numpy as np
import pytest
import torch

from tests import ep_harness as HN
from tests.test_parity_gpu import _routing, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


WIDE = {
    # name: (T, K, E, R, H, M, A, expand, zero_pad, sync, fp8, col_major, drop, form)
    # form: 1 = the cluster kernel (rank layout, at most 15 chunks), 2 = the
    # count and assign kernels
    # 33..64 ranks: the 64-bit mask walk (R % 4 == 0: packed rank rows)
    "r48_rank_fp8_sync": (2000, 8, 192, 48, 256, 300, 1, False, False, True, True, False, 0.05, 1),
    "r48_expand_bf16_nosync": (2000, 8, 192, 48, 256, 300, 4, True, True, False, False, False, 0.0, 2),
    "r50_rank_bf16_nosync": (1500, 6, 100, 50, 128, 37, 1, False, False, False, False, False, 0.1, 2),
    "r50_expand_fp8cm_sync": (1500, 6, 100, 50, 256, 37, 8, True, True, True, True, True, 0.1, 2),
    "r64_rank_fp8_nosync": (2000, 8, 256, 64, 512, 300, 1, False, False, False, True, False, 0.0, 1),
    "r64_expand_fp8cm_sync": (2000, 8, 256, 64, 256, 300, 16, True, True, True, True, True, 0.02, 2),
    # more than 64 ranks: look-back rank sets, byte-wise rank rows
    "r100_rank_bf16_sync": (2000, 8, 300, 100, 128, 20, 1, False, False, True, False, False, 0.05, 2),
    "r128_rank_bf16_cluster": (2000, 8, 256, 128, 256, 300, 1, False, False, True, False, False,
                               0.05, 1),
    "r128_rank_fp8_sync": (3000, 8, 256, 128, 256, 24, 1, False, False, True, True, False, 0.0, 2),
    "r128_expand_bf16_nosync": (3000, 8, 256, 128, 128, 300, 8, True, True, False, False, False, 0.05, 2),
    "r256_rank_fp8_nosync": (2000, 8, 256, 256, 256, 9, 1, False, False, False, True, False, 0.0, 2),
    "r256_rank_bf16_sync": (2000, 8, 256, 256, 128, 300, 1, False, False, True, False, False, 0.02, 1),
    "r256_expand_fp8cm_sync": (2000, 8, 256, 256, 256, 9, 8, True, True, True, True, True, 0.0, 2),
    "r256_expand_fp8_nosync": (2000, 8, 256, 256, 256, 300, 4, True, True, False, True, False, 0.1, 2),
}


@pytest.mark.parametrize("case", sorted(WIDE))
def test_wide_rank_parity(ep, case):
    T, K, E, R, H, M, A, ex, zp, sync, fp8, cm, drop, form = WIDE[case]
    assert T <= M * R
    idx, w = _routing(T, K, E, seed=zlib.crc32(case.encode()) % 1000, drop=drop)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, A, ex, zp, sync, fp8, cm)
    r = run_and_check(ep, cfg, idx, x, w, bias0=True)
    assert r["combine_mismatch"] == 0
    assert r["layout_kernels"] == form
    lay = r["lay"]
    # every rank is reached, so every rank-set branch wrote rows
    assert int((lay["cnt_rank"] > 0).sum()) == R


def test_wide_rank_unweighted_combine(ep):
    """Rank layout at 128 ranks without weights: a token's slots on one rank
    share a row, which the combine must count once."""
    T, K, E, R, H, M = 1200, 8, 256, 128, 256, 10
    idx, w = _routing(T, K, E, seed=31, drop=0.05, dup=True)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 1, False, False, True)
    r = run_and_check(ep, cfg, idx, x, w, combine_w=False)
    assert r["combine_mismatch"] == 0


def test_ep256_decode_full_size(ep):
    """A full 256-rank decode batch: 128 tokens per rank (32768 tokens),
    hidden 7168, 256 experts (one per rank), top-8, FP8 with row-major
    scales, rank layout, upper-bound allocation.  Every layout output is
    compared in full; dispatch and combine on 256 sampled tokens."""
    T, K, E, R, H, M = 32768, 8, 256, 256, 7168, 128
    idx, w = _routing(T, K, E, seed=41)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    cfg = ep.make_config(T, K, E, R, H, M, 1, False, False, False, True, False)
    toks = np.sort(np.random.default_rng(3).choice(T, size=256, replace=False))
    r = run_and_check(ep, cfg, idx, x, w, combine_tokens=toks, dispatch_tokens=toks)
    assert r["combine_mismatch"] == 0
    assert r["lay"]["rows_alloc"] == T * K
