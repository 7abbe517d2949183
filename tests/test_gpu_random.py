"""Randomised GPU parity: seeded random problems across the supported space
(K/V dtype, D, group size, page size, batch, length mix, split count, stage
tile, CTAs per SM, fused or separate merge, output dtype), each compared with
the fp64 oracle on every row at the bars of the other parity tests.  Sized so
the oracle finishes each in well under a second."""
import numpy as np
import pytest
import torch

from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, gpu_decode, oracle_full

pytestmark = pytest.mark.gpu


def _draw(rng):
    kv = str(rng.choice(["f16", "bf16", "e4m3"]))
    q = "f16" if kv == "f16" else str(rng.choice(["bf16", "f16"])) if kv == "e4m3" else "bf16"
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 5, 8, 12, 16]))
    ps = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.choice([1, 2, 3, 7, 40]))
    maxL = int(rng.choice([1, 37, 300, 1500, 6000]))
    lens = rng.integers(0, maxL + 1, B)
    lens[0] = maxL
    opts = {}
    r = rng.random()
    if r < 0.2:
        opts["num_splits"] = int(rng.choice([1, 2, 3, 8, 17]))
    elif r < 0.3:
        opts["tile_tokens"] = 64
        opts["ctas_per_sm"] = 2
    elif r < 0.4:
        opts["fuse_merge"] = 0
        opts["num_splits"] = int(rng.choice([2, 5]))
    out_dtype = torch.float32 if rng.random() < 0.5 else None
    spec = W.Spec(f"random {kv}/{q} D={D} G={G} Hkv={Hkv} ps={ps} B={B}", B=B, Hq=Hkv * G, Hkv=Hkv, D=D,
                  page_size=ps, kv=kv, q=q, lens=("list", lens.tolist()), pool=("factor", 1.5))
    return spec, opts, out_dtype


@pytest.mark.parametrize("seed", range(48))
def test_random_problem_matches_oracle(fdlib, seed):
    rng = np.random.default_rng(9000 + seed)
    spec, opts, out_dtype = _draw(rng)
    wl = W.make(spec, 500 + seed, "cpu")
    try:
        out, lse, dec = gpu_decode(wl.to("cuda"), out_dtype=out_dtype, **opts)
    except Exception as e:  # a shape the plan options do not allow (e.g. two CTAs that do not fit)
        from split_kv_decode_paged_gb300._lib import FdError, FD_ERR_UNSUPPORTED
        if isinstance(e, FdError) and e.code == FD_ERR_UNSUPPORTED and opts:
            pytest.skip(f"options {opts} unsupported for {spec.name}")
        raise
    ref_o, ref_l = oracle_full(wl)
    assert_close(spec.kv, out, lse, ref_o, ref_l, what=f"{spec.name} {opts} out={out_dtype}")


@pytest.mark.parametrize("seed", range(16))
def test_random_multi_token_problem_matches_oracle(fdlib, seed):
    """Several causal query tokens per sequence on random problems: q_len in
    2..8, lengths at least q_len, random split count and merge mode."""
    from tests.test_gpu_multi import _run
    rng = np.random.default_rng(7000 + seed)
    kv = str(rng.choice(["f16", "bf16", "e4m3"]))
    q = "f16" if kv == "f16" else "bf16"
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    q_len = int(rng.integers(2, 9))
    ps = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.choice([1, 2, 5, 12]))
    lens = rng.integers(q_len, int(rng.choice([q_len + 1, 200, 2500])) + 1, B).tolist()
    splits = int(rng.choice([0, 0, 2, 5]))
    fuse = int(rng.random() < 0.7)
    _run(kv, q, ps, D, Hkv * G, Hkv, q_len, lens, seed=300 + seed, out32=bool(rng.random() < 0.5),
         num_splits=splits, fuse_merge=fuse)
