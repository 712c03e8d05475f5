"""GPU parity on a seeded sweep of random configurations, against the oracle.

The hand-picked cases elsewhere pin each branch on purpose; this sweep draws
the combinations they do not name: rank counts from 1 to 128 with 1 to 32
experts per rank, top-k from 1 to 32, hidden sizes from 8 to 7168, BF16 and
FP8 with both scale layouts, the rank, expanded (with and without zero
padding, alignments up to 128) and fixed-capacity layouts, with and without
the host count wait, empty slots, repeated experts, token counts from 0 to
the per-rank maximum, and both entry points (ep_layout + ep_dispatch, and
ep_layout_dispatch where there is no count wait).  Every configuration is
kept only if ep_validate_config accepts it.  Layout, metadata and dispatch
bytes must match bit for bit; combine within 1 BF16 ulp (and in practice
exactly), weighted with a per-token bias, or unweighted.
"""
import numpy as np
import pytest
import torch

from tests.test_parity_gpu import _routing, run_and_check

pytestmark = pytest.mark.gpu

N_CASES = 96
MAX_ELEMS = 12_000_000  # T * K * H, so that the oracle finishes in about a second
MAX_Y_ELEMS = 64 << 20  # rows of the upper-bound allocation * H


def _draw(ep, rng):
    """One random configuration accepted by ep_validate_config, as kwargs."""
    while True:
        R = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 48, 64, 128]))
        L = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
        E = R * L
        if E > 2048:
            continue
        K = int(rng.integers(1, min(E, 32) + 1))
        fp8 = bool(rng.random() < 0.5)
        H = int(rng.choice([128, 256, 384, 1024, 7168] if fp8 else [8, 64, 136, 256, 520, 2048]))
        M = int(rng.integers(1, 300))
        t_cap = min(M * R, 2500, MAX_ELEMS // (K * H))
        T = int(rng.integers(0, t_cap + 1))
        expand = bool(rng.random() < 0.5)
        fixed = expand and bool(rng.random() < 0.25)
        A = 1 if (not expand or fixed) else int(rng.choice([1, 2, 4, 8, 16, 32, 128]))
        zp = expand and not fixed and bool(rng.random() < 0.7)
        sync = bool(rng.random() < 0.5)
        cm = fp8 and bool(rng.random() < 0.5)
        drop = float(rng.choice([0.0, 0.05, 0.3]))
        dup = bool(rng.random() < 0.15)
        fused = not sync and bool(rng.random() < 0.6)
        weighted = bool(rng.random() < 0.8)
        cfg = ep.make_config(T, K, E, R, H, M, A, expand, zp, sync, fp8, cm,
                             fixed_capacity=fixed)
        if ep.validate_config(cfg) != ep.EP_OK:
            continue
        if ep.upper_bound_rows(cfg) * H > MAX_Y_ELEMS:  # y and its oracle copy stay small
            continue
        return dict(T=T, K=K, E=E, R=R, H=H, M=M, A=A, expand=expand, zp=zp, sync=sync,
                    fp8=fp8, cm=cm, fixed=fixed, drop=drop, dup=dup, fused=fused,
                    weighted=weighted)


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


@pytest.fixture(scope="module")
def cases(ep):
    rng = np.random.default_rng(20261203)
    return [_draw(ep, rng) for _ in range(N_CASES)]


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_config_parity(ep, cases, i):
    c = cases[i]
    idx, w = _routing(c["T"], c["K"], c["E"], seed=1000 + i, drop=c["drop"], dup=c["dup"])
    x = torch.randn(c["T"], c["H"], generator=torch.Generator().manual_seed(2000 + i))
    x = x.to(torch.bfloat16)
    cfg = ep.make_config(c["T"], c["K"], c["E"], c["R"], c["H"], c["M"], c["A"], c["expand"],
                         c["zp"], c["sync"], c["fp8"], c["cm"], fixed_capacity=c["fixed"])
    r = run_and_check(ep, cfg, idx, x, w, bias0=c["weighted"], combine_w=c["weighted"],
                      fused=c["fused"])
    assert r["combine_mismatch"] == 0, c
