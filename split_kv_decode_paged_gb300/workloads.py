"""Seeded synthetic decode workloads: paged K/V pools, block tables, lengths.

This module only draws inputs; it holds none of the attention arithmetic.
Both the CUDA path and the CPU oracle consume the tensors it returns, so a
value stream may differ between devices (a CUDA generator and a CPU generator
give different numbers for one seed) without affecting parity: both sides
always see the same stored tensors.

Layout (FlashAttention "Inference Cookbook", §4.2): K and V pools are
[num_pages, page_size, Hkv, D]; the block table is int32 [B, max_blocks]
with -1 in unused entries; seq_lens is int32 [B].  Pages not referenced by
any sequence and slots past a sequence's length are filled with NaN so that
a wrong gather shows up in the output.

FP8 pools (E4M3) carry one fp32 scale per (page, KV head): the values are
drawn in fp32, the scale is the page's max |x| over its live slots divided
by 448 (floored at 1e-12), and the stored code is x / scale rounded by
torch's float8_e4m3fn conversion.  Unused pages get NaN codes and NaN scales.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0
_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn,
       "f32": torch.float32}


@dataclass
class Spec:
    """One synthetic decode workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    kv: str                      # "f16" | "bf16" | "e4m3"
    q: str                       # "f16" | "bf16"
    lens: tuple                  # ("const", L) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    pool: tuple = ("factor", 1.0)  # ("identity",) | ("factor", f): pool = f * needed pages
    k_mult: float = 1.0          # K ~ k_mult * N(0, 1)
    extra_blocks: int = 0        # spare block-table columns (append capacity)
    splits: list = field(default_factory=list)  # forced split counts used by parity tests


# The five workloads (shapes, dtypes, length mixes and page pools).
CONFIGS = {
    1: Spec("tiny MHA decode", B=1, Hq=4, Hkv=4, D=64, page_size=16, kv="f16", q="f16",
            lens=("const", 256), pool=("identity",), splits=[1, 4]),
    2: Spec("single-sequence MHA split-KV", B=1, Hq=32, Hkv=32, D=128, page_size=16, kv="f16",
            q="f16", lens=("const", 4096), pool=("factor", 2.0)),
    3: Spec("Llama-3-8B-shaped GQA batch", B=64, Hq=32, Hkv=8, D=128, page_size=16, kv="bf16",
            q="bf16", lens=("uniform", 512, 8192), pool=("factor", 1.1)),
    4: Spec("long-context single request", B=1, Hq=32, Hkv=8, D=128, page_size=64, kv="bf16",
            q="bf16", lens=("const", 131072), pool=("factor", 2.0), k_mult=2.0),
    5: Spec("mixed serving batch, large pages, FP8 cache", B=256, Hq=64, Hkv=8, D=128,
            page_size=128, kv="e4m3", q="bf16", lens=("loguniform", 16, 32768),
            pool=("factor", 1.1)),
}


# Two large batches beyond the five workloads (many 32-row blocks of the
# dispatch tables): short bf16 contexts, and an FP8 cache with a wide length mix.
LARGE_BATCHES = {
    "bf16 B=1024": Spec("large GQA batch, short contexts", B=1024, Hq=32, Hkv=8, D=128, page_size=16, kv="bf16",
                        q="bf16", lens=("uniform", 256, 1024), pool=("factor", 1.1)),
    "e4m3 B=2048": Spec("large FP8 batch, mixed lengths", B=2048, Hq=32, Hkv=8, D=128, page_size=64, kv="e4m3",
                        q="bf16", lens=("loguniform", 16, 4096), pool=("factor", 1.1)),
}
LARGE_BATCH_SEED = 77


def config_seed(cfg_id: int) -> int:
    return 1000 + int(cfg_id)


def draw_lengths(spec: Spec, gen: torch.Generator) -> torch.Tensor:
    kind = spec.lens[0]
    if kind == "const":
        return torch.full((spec.B,), int(spec.lens[1]), dtype=torch.int32)
    if kind == "uniform":
        lo, hi = spec.lens[1], spec.lens[2]
        return torch.randint(lo, hi + 1, (spec.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        lo, hi = math.log(spec.lens[1]), math.log(spec.lens[2])
        u = torch.rand((spec.B,), generator=gen, dtype=torch.float64)
        return torch.round(torch.exp(lo + (hi - lo) * u)).to(torch.int32)
    if kind == "list":
        return torch.tensor(list(spec.lens[1]), dtype=torch.int32)
    raise ValueError(kind)


@dataclass
class Workload:
    spec: Spec
    q: torch.Tensor            # [B, Hq, D]
    k_pages: torch.Tensor      # [num_pages, page_size, Hkv, D]
    v_pages: torch.Tensor
    k_scale: torch.Tensor | None  # [num_pages, Hkv] fp32 (E4M3 only)
    v_scale: torch.Tensor | None
    block_table: torch.Tensor  # [B, max_blocks] int32
    seq_lens: torch.Tensor     # [B] int32 (host copy, same values)
    num_pages: int

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def to(self, device) -> "Workload":
        mv = lambda t: None if t is None else t.to(device)
        return Workload(self.spec, mv(self.q), mv(self.k_pages), mv(self.v_pages),
                        mv(self.k_scale), mv(self.v_scale), mv(self.block_table),
                        mv(self.seq_lens), self.num_pages)


def _fill_pool(pool: torch.Tensor, live: torch.Tensor, gen: torch.Generator, mult: float,
               chunk: int = 1024) -> None:
    """Draw N(0,1)*mult into pool (fp16/bf16), page chunk by page chunk; NaN
    where live is False ([num_pages, page_size] mask)."""
    n = pool.shape[0]
    for p0 in range(0, n, chunk):
        p1 = min(n, p0 + chunk)
        x = torch.randn(pool[p0:p1].shape, generator=gen, dtype=torch.float32, device=pool.device)
        if mult != 1.0:
            x.mul_(mult)
        m = live[p0:p1]
        x[~m] = float("nan")
        pool[p0:p1].copy_(x.to(pool.dtype))


def _fill_pool_fp8(pool: torch.Tensor, scale: torch.Tensor, live: torch.Tensor,
                   gen: torch.Generator, mult: float, chunk: int = 1024) -> None:
    n = pool.shape[0]
    for p0 in range(0, n, chunk):
        p1 = min(n, p0 + chunk)
        x = torch.randn(pool[p0:p1].shape, generator=gen, dtype=torch.float32, device=pool.device)
        if mult != 1.0:
            x.mul_(mult)
        m = live[p0:p1]                                    # [P, page_size]
        mm = m[:, :, None, None].expand_as(x)
        amax = torch.where(mm, x.abs(), torch.zeros_like(x)).amax(dim=(1, 3))  # [P, Hkv]
        sc = torch.clamp(amax / E4M3_MAX, min=1e-12)
        any_live = m.any(dim=1)                            # [P]
        sc[~any_live] = float("nan")
        y = x / sc[:, None, :, None]
        y = torch.clamp(y, -E4M3_MAX, E4M3_MAX)
        codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
        codes[~mm] = 0x7F                                  # NaN code
        pool[p0:p1].view(torch.uint8).copy_(codes)
        scale[p0:p1].copy_(sc)


def make(spec: Spec, seed: int, device="cpu", seq_lens=None) -> Workload:
    """Draw a workload.  seq_lens (list/tensor) overrides the spec's length mix."""
    device = torch.device(device)
    g_host = torch.Generator().manual_seed(int(seed))
    lens = (torch.as_tensor(seq_lens, dtype=torch.int32).cpu() if seq_lens is not None
            else draw_lengths(spec, g_host))
    ps = spec.page_size
    npages_seq = [max(0, (int(L) + ps - 1) // ps) for L in lens.tolist()]
    needed = sum(npages_seq)
    max_blocks = max([1] + npages_seq) + spec.extra_blocks
    if spec.pool[0] == "identity":
        num_pages = max(1, needed + spec.extra_blocks * spec.B)
        perm = torch.arange(num_pages, dtype=torch.int32)
    else:
        num_pages = max(1, int(math.ceil(needed * float(spec.pool[1]))) + spec.extra_blocks * spec.B)
        perm = torch.randperm(num_pages, generator=g_host).to(torch.int32)
    bt = torch.full((spec.B, max_blocks), -1, dtype=torch.int32)
    live = torch.zeros((num_pages, ps), dtype=torch.bool)
    cur = 0
    for b, n in enumerate(npages_seq):
        pages = perm[cur:cur + n]
        cur += n
        bt[b, :n] = pages
        L = int(lens[b])
        for j in range(n):
            live[int(pages[j]), : min(ps, L - j * ps)] = True
    # Spare columns (append capacity) take further pool pages in order.
    if spec.extra_blocks:
        for b in range(spec.B):
            for j in range(spec.extra_blocks):
                bt[b, npages_seq[b] + j] = perm[cur]
                cur += 1

    g_dev = torch.Generator(device=device).manual_seed(int(seed) + 1)
    shape = (num_pages, ps, spec.Hkv, spec.D)
    live_dev = live.to(device)
    if spec.kv == "e4m3":
        kp = torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)
        vp = torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)
        ks = torch.empty((num_pages, spec.Hkv), dtype=torch.float32, device=device)
        vs = torch.empty((num_pages, spec.Hkv), dtype=torch.float32, device=device)
        _fill_pool_fp8(kp, ks, live_dev, g_dev, spec.k_mult)
        _fill_pool_fp8(vp, vs, live_dev, g_dev, 1.0)
    else:
        kp = torch.empty(shape, dtype=_DT[spec.kv], device=device)
        vp = torch.empty(shape, dtype=_DT[spec.kv], device=device)
        ks = vs = None
        _fill_pool(kp, live_dev, g_dev, spec.k_mult)
        _fill_pool(vp, live_dev, g_dev, 1.0)
    q = torch.randn((spec.B, spec.Hq, spec.D), generator=g_dev, dtype=torch.float32,
                    device=device).to(_DT[spec.q])
    return Workload(spec, q, kp, vp, ks, vs, bt.to(device), lens.to(device), num_pages)


def make_config(cfg_id: int, device="cpu", seed=None) -> Workload:
    return make(CONFIGS[cfg_id], config_seed(cfg_id) if seed is None else seed, device)


def algorithmic_bytes(spec: Spec, seq_lens, out_bytes_per_elem=None) -> int:
    """Bytes one decode call must move: K+V of the live tokens, q, out, lse,
    the live block-table entries, seq_lens and (FP8) the live pages' scales."""
    e = 1 if spec.kv == "e4m3" else 2
    eq = 4 if spec.q == "f32" else 2
    eo = eq if out_bytes_per_elem is None else out_bytes_per_elem
    lens = [int(x) for x in (seq_lens.tolist() if hasattr(seq_lens, "tolist") else seq_lens)]
    tok = sum(lens)
    pages = sum((L + spec.page_size - 1) // spec.page_size for L in lens)
    n = tok * spec.Hkv * spec.D * 2 * e
    n += spec.B * spec.Hq * spec.D * (eq + eo) + 4 * spec.B * spec.Hq
    n += 4 * pages + 4 * spec.B
    if spec.kv == "e4m3":
        n += 2 * 4 * spec.Hkv * pages
    return n


@dataclass
class SharedPrefixWorkload:
    """A batch whose sequences share their first prefix_len tokens (whole
    pages, stored once) and then continue with their own tokens."""
    flat: Workload               # per-sequence tables: prefix pages, then own pages
    prefix_table: torch.Tensor   # [1, prefix_blocks]
    prefix_len: int
    suffix_table: torch.Tensor   # [B, suffix_max_blocks]
    suffix_lens: torch.Tensor    # [B]


def make_shared_prefix(spec: Spec, seed: int, prefix_len: int, suffix_lens, device="cpu") -> SharedPrefixWorkload:
    """Draw a shared-prefix batch: spec gives the shapes and dtypes (its
    length mix is ignored); the pool holds the prefix pages once."""
    ps = spec.page_size
    if prefix_len % ps:
        raise ValueError("prefix_len must be a multiple of page_size")
    suffix = torch.as_tensor(suffix_lens, dtype=torch.int32)
    B = spec.B
    n_pre = prefix_len // ps
    n_suf = [(int(L) + ps - 1) // ps for L in suffix.tolist()]
    flat_lens = suffix + prefix_len
    # Draw one pool sized for the prefix once plus every suffix, as a flat
    # workload whose sequence 0 holds the prefix; then rewrite the tables.
    total_pages = n_pre + sum(n_suf)
    base = make(Spec(spec.name, B=1, Hq=spec.Hq, Hkv=spec.Hkv, D=spec.D, page_size=ps, kv=spec.kv, q=spec.q,
                     lens=("list", [total_pages * ps]), pool=("factor", 1.0)), seed, device)
    pages = base.block_table[0].cpu()
    prefix_pages = pages[:n_pre]
    max_suf = max([1] + n_suf)
    suffix_table = torch.full((B, max_suf), -1, dtype=torch.int32)
    flat_table = torch.full((B, n_pre + max_suf), -1, dtype=torch.int32)
    cur = n_pre
    for b in range(B):
        own = pages[cur:cur + n_suf[b]]
        cur += n_suf[b]
        suffix_table[b, :n_suf[b]] = own
        flat_table[b, :n_pre] = prefix_pages
        flat_table[b, n_pre:n_pre + n_suf[b]] = own
    g = torch.Generator(device=torch.device(device)).manual_seed(int(seed) + 7)
    q = torch.randn((B, spec.Hq, spec.D), generator=g, dtype=torch.float32, device=device).to(_DT[spec.q])
    dspec = Spec(spec.name, B=B, Hq=spec.Hq, Hkv=spec.Hkv, D=spec.D, page_size=ps, kv=spec.kv, q=spec.q,
                 lens=("list", flat_lens.tolist()))
    flat = Workload(dspec, q, base.k_pages, base.v_pages, base.k_scale, base.v_scale, flat_table.to(device),
                    flat_lens.to(device), base.num_pages)
    return SharedPrefixWorkload(flat, prefix_pages.view(1, -1).to(device), prefix_len, suffix_table.to(device),
                                suffix.to(device))
