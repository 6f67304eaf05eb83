"""Host-side page bookkeeping for the mixed cache: page tables, prefix sharing and
pool allocation.  The library itself never allocates; this is the caller-side
allocator the tests and the benchmark use (a serving system would bring its
own).  Physical page ids are handed out in order; a shared prefix maps the
first pages of every sequence to the same physical ids.
"""
from __future__ import annotations

import dataclasses

import numpy as np

PAGE = 16


def int2_page_needed(p: int, L: int, sink: int, window: int) -> bool:
    """Logical page p holds a token of the INT2 region [sink, L - window)."""
    return p * PAGE < L - window and p * PAGE + PAGE > sink


def bf16_page_needed(p: int, L: int, sink: int, window: int) -> bool:
    lo, hi = p * PAGE, min(p * PAGE + PAGE, L)
    return lo < hi and (lo < sink or hi > L - window)


@dataclasses.dataclass
class PagePlan:
    int2_table: np.ndarray      # int32 [B, max_pages]
    bf16_table: np.ndarray
    num_int2_pages: int
    num_bf16_pages: int
    max_pages: int


def plan(seq_lens, sink: int, window: int, *, shared_prefix_tokens: int = 0,
         max_len: int | None = None, growth: int = 0, all_pages: bool = False,
         permute_seed: int | None = None) -> PagePlan:
    """Allocate pages for sequences of the given final lengths.

    growth: extra decode steps to provision for (the window slides, so INT2
    pages are allocated up to L + growth - window and BF16 pages up to L +
    growth).  all_pages: give every logical page both kinds.  permute_seed:
    shuffle physical ids (to show placement does not matter).  Pages wholly
    inside the shared prefix are shared by all sequences.
    """
    lens = np.asarray(seq_lens, np.int64)
    B = len(lens)
    top = int(lens.max()) + growth if max_len is None else max_len
    maxp = (top + PAGE - 1) // PAGE
    it = np.full((B, maxp), -1, np.int32)
    bt = np.full((B, maxp), -1, np.int32)
    n2 = nb = 0
    shared = shared_prefix_tokens // PAGE
    shared2, sharedb = {}, {}
    for b in range(B):
        L0, L1 = int(lens[b]), int(lens[b]) + growth
        for p in range((L1 + PAGE - 1) // PAGE):
            # INT2 region only grows with the length; the BF16 window slides
            # over [L0 - window, L1) while appending
            need2 = all_pages or int2_page_needed(p, L1, sink, window)
            needb = all_pages or p * PAGE < sink or (p * PAGE + PAGE > L0 - window and p * PAGE < L1)
            if p < shared:
                if need2:
                    if p not in shared2:
                        shared2[p] = n2
                        n2 += 1
                    it[b, p] = shared2[p]
                if needb:
                    if p not in sharedb:
                        sharedb[p] = nb
                        nb += 1
                    bt[b, p] = sharedb[p]
                continue
            if need2:
                it[b, p] = n2
                n2 += 1
            if needb:
                bt[b, p] = nb
                nb += 1
    if permute_seed is not None:
        rng = np.random.default_rng(permute_seed)
        p2 = rng.permutation(max(n2, 1)).astype(np.int32)
        pb = rng.permutation(max(nb, 1)).astype(np.int32)
        it = np.where(it >= 0, p2[np.maximum(it, 0)], -1).astype(np.int32)
        bt = np.where(bt >= 0, pb[np.maximum(bt, 0)], -1).astype(np.int32)
    return PagePlan(it, bt, max(n2, 1), max(nb, 1), maxp)


def int2_bytes_per_page(hkv: int, d: int, code_bits: int = 2) -> int:
    """Code-pool bytes of one page: 12d per KV head for INT2, 20d for the INT4
    variant (two 2-bit planes)."""
    return hkv * (4 * code_bits + 4) * d


def bf16_bytes_per_page(hkv: int, d: int) -> int:
    return hkv * 64 * d


def allocate(pp: PagePlan, *, hkv: int, hq: int, d: int, sink: int, window: int, device,
             r_k=None, r_v=None, clip_k=None, clip_v=None, with_status: bool = True,
             code_bits: int = 2):
    """Device pools (zeroed) and tables for a plan; returns a binding ``Cache``.
    code_bits: 2 (INT2 pages) or 4 (the INT4 variant)."""
    import torch

    from ._lib import Cache
    dev = torch.device(device)
    int2 = torch.zeros(pp.num_int2_pages * int2_bytes_per_page(hkv, d, code_bits), dtype=torch.uint8,
                       device=dev)
    bf = torch.zeros(pp.num_bf16_pages * hkv * 32 * d, dtype=torch.bfloat16, device=dev)

    def t(x, dt):
        return None if x is None else torch.as_tensor(np.ascontiguousarray(x), dtype=dt).to(dev)

    return Cache(hkv, hq, d, sink, window, int2, bf,
                 t(pp.int2_table, torch.int32), t(pp.bf16_table, torch.int32),
                 t(r_k, torch.float32), t(r_v, torch.float32), t(clip_k, torch.float32),
                 t(clip_v, torch.float32),
                 torch.zeros(1, dtype=torch.int32, device=dev) if with_status else None, code_bits)
