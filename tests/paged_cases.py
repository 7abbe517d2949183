"""Small hand-built paged caches for oracle pins.

Builds a paged pool from per-token contiguous arrays by scattering each
token to (page, slot) under a random page permutation, independently of the
oracle's gather.  Values are chosen exactly representable in the storage
dtype so that expected values can be computed from the float arrays.
"""
import numpy as np
import torch

from oracle import oracle as orc

_TORCH = {orc.F16: torch.float16, orc.BF16: torch.bfloat16, orc.F32: torch.float32}


def to_storage(x: np.ndarray, code: int) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, np.float64)).to(_TORCH[code])
    back = t.to(torch.float64).numpy()
    assert np.array_equal(back, x, equal_nan=True), "values must be exact in the storage dtype"
    return t


def round_to(x: np.ndarray, code: int) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float64)).to(_TORCH[code]).to(torch.float64).numpy()


def build_paged(K, V, lens, page_size, rng, spare_pages=3, kv_code=orc.F32):
    """K, V: float arrays [B, Lmax, Hkv, D].  Returns (k_pages, v_pages,
    block_table, num_pages) with pages scattered by a random permutation and
    spare (unreferenced) pages filled with NaN."""
    B, Lmax, Hkv, D = K.shape
    npg = [(int(L) + page_size - 1) // page_size for L in lens]
    num_pages = sum(npg) + spare_pages
    perm = rng.permutation(num_pages)
    kp = np.full((num_pages, page_size, Hkv, D), np.nan)
    vp = np.full((num_pages, page_size, Hkv, D), np.nan)
    max_blocks = max([1] + npg)
    bt = np.full((B, max_blocks), -1, np.int32)
    cur = 0
    for b in range(B):
        for j in range(npg[b]):
            bt[b, j] = perm[cur]
            cur += 1
        for t in range(int(lens[b])):
            page, slot = bt[b, t // page_size], t % page_size
            kp[page, slot] = K[b, t]
            vp[page, slot] = V[b, t]
    return to_storage(kp, kv_code), to_storage(vp, kv_code), bt, num_pages
