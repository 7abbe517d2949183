"""Randomised host-side checks of fd_plan (no GPU): for a few hundred seeded
problems -- valid and invalid dimensions, dtypes, page sizes, length mixes,
split and shape options -- the planner either rejects the problem with a
status code or returns a plan whose fields satisfy the invariants the kernel
relies on.  Nothing may crash, and the same inputs give the same plan."""
import numpy as np
import pytest
import torch

from split_kv_decode_paged_gb300 import _lib

SMEM_OPTIN = 232448
SM_SMEM, RESERVED = 233472, 1024
KV = [torch.float16, torch.bfloat16, torch.float8_e4m3fn]


def _draw(rng):
    D = int(rng.choice([64, 128, 96, 256]))            # 96 and 256 are unsupported
    Hkv = int(rng.choice([1, 2, 4, 8, 16]))
    G = int(rng.choice([1, 2, 3, 4, 8, 12, 16, 20, 32]))
    Hq = Hkv * G if rng.random() > 0.05 else Hkv * G + 1   # a few Hq % Hkv != 0
    ps = int(rng.choice([16, 32, 64, 128, 8, 24]))      # 8 and 24 are not multiples of 16
    B = int(rng.choice([1, 2, 5, 64, 300, 2048]))
    kv = KV[int(rng.integers(len(KV)))]
    q = torch.float16 if kv == torch.float16 else torch.bfloat16
    maxL = int(rng.choice([1, 100, 1000, 5000, 40000]))
    mix = int(rng.integers(3))
    if mix == 0:
        lens = [maxL] * B
    elif mix == 1:
        lens = rng.integers(0, maxL + 1, B).tolist()
    else:
        lens = np.minimum(np.exp(rng.uniform(0, np.log(maxL + 1), B)).astype(int), maxL).tolist()
    mb = (maxL + ps - 1) // ps + int(rng.integers(0, 3))
    opts = {}
    r = rng.random()
    if r < 0.15:
        opts["num_splits"] = int(rng.choice([1, 2, 7, 64, 600]))
    elif r < 0.25:
        opts["tile_tokens"] = int(rng.choice([64, 128, 256, 96]))
    elif r < 0.35:
        opts["ctas_per_sm"] = int(rng.choice([1, 2, 3]))
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, ps=ps, mb=mb, kv=kv, q=q), lens, opts


@pytest.mark.parametrize("seed", range(6))
def test_random_problems_plan_or_reject(fdlib, seed):
    rng = np.random.default_rng(1234 + seed)
    planned = 0
    for _ in range(60):
        d, lens, opts = _draw(rng)
        prob = _lib.make_problem(d["B"], d["Hq"], d["Hkv"], d["D"], d["ps"], d["mb"], d["B"] * d["mb"] + 1,
                                 d["q"], d["kv"])
        try:
            plan = _lib.fd_plan(prob, lens, num_sms=152, **opts)
        except _lib.FdError as e:
            assert e.code in (_lib.FD_ERR_INVALID_ARG, _lib.FD_ERR_UNSUPPORTED), (d, opts, e)
            continue
        planned += 1
        # the problem was valid
        assert d["D"] in (64, 128) and d["ps"] % 16 == 0 and d["Hq"] % d["Hkv"] == 0
        # the kernel's invariants
        assert plan.tile_tokens in (64, 128, 256) and plan.chunk_tokens % plan.tile_tokens == 0
        assert plan.capacity_tokens >= max(lens) and plan.capacity_tokens == plan.num_splits * plan.chunk_tokens
        assert 1 <= plan.num_splits <= 512
        cps = max(1, plan.ctas_per_sm)
        assert (cps in (1, 2) or opts.get("ctas_per_sm") == cps) and 1 <= plan.grid_ctas <= 152 * cps
        limit = SMEM_OPTIN if cps == 1 else (SM_SMEM - cps * RESERVED) // cps
        assert 2 <= plan.stages <= 8 and plan.smem_bytes <= limit
        G = d["Hq"] // d["Hkv"]
        qrows = 16 if G > 8 else 8
        assert plan.head_subgroups == (G + qrows - 1) // qrows
        items = sum((1 if L == 0 else (L + plan.chunk_tokens - 1) // plan.chunk_tokens) for L in lens)
        assert plan.work_items_hint == items * d["Hkv"] * plan.head_subgroups
        rows = d["B"] * d["Hq"]
        if plan.num_splits > 1:
            assert plan.workspace_bytes >= rows * plan.num_splits * (d["D"] + 2) * 4
        # deterministic
        again = _lib.fd_plan(prob, lens, num_sms=152, **opts)
        assert bytes(again) == bytes(plan)
    assert planned >= 10
