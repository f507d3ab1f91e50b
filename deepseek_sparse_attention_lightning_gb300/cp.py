"""Context-parallel decode: one long request's cached tokens split over ranks.

Each rank holds a contiguous, page-aligned slice of every request's cached
tokens -- its own part of the index-key cache and of the latent cache, with
its own page table -- and the (replicated) queries.  One decode layer is
three phases with an exchange after each of the first two:

  A  score the local slice (lightning indexer over local positions) and take
     its local top-k; the candidates are the local winners' scores and their
     global positions (a local winner set contains every global winner that
     lies in the slice, since a token beaten by k tokens of its own slice is
     beaten by k tokens of the request);
  -- all-gather the candidates (k scores and k positions per query and rank);
  B  the global top-k over the R * k candidates (ties go to the lower global
     position: the ranks' lists are concatenated in slice order and each is
     ascending, so a lower candidate index is a lower position), then the
     sparse attention over the winners this rank holds, one split: a partial
     output and its log-sum-exp;
  -- all-gather the partials;
  C  the merge of the R partials (the split-KV merge with one split per rank).

This is the exchange step of "Deepseek Details", section "DSA" (stages 2-3:
split partials and their merge) applied across ranks, with the selection of
"MTP and sparse attention: NSA and DSA", section "Sparse attention: NSA and
DSA" (each query keeps its k best tokens) made global by a second top-k over
the ranks' local winners.  The pages name context-parallel splitting only
("[SGLang] NSA", its module list); this layout is the library's.

Every step on a rank runs in the library's kernels (``DeviceSteps``); the
exchanges are ``torch.distributed`` all-gathers (NCCL between GPUs, gloo in
the CPU tests, which inject their own steps), or, with ``run_emulated``, the
concatenation of R slices processed one after another in this process.
Remote data is always copied into local memory first.  Query tokens per
request must be 1 (each slice is then a plain request of its own length).
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence

import torch

from . import api

PAGE = api.PAGE_SIZE


def slice_bounds(seqlen: int, ranks: int) -> List[int]:
    """Page-aligned bounds b[0] = 0 < ... <= b[ranks] = seqlen of the ranks'
    contiguous slices of a request of `seqlen` tokens (the last slice takes
    the ragged tail; a slice may be empty when the request is short)."""
    if ranks < 1 or seqlen < 0:
        raise ValueError("ranks >= 1 and seqlen >= 0")
    pages = (seqlen + PAGE - 1) // PAGE
    b = [min(seqlen, ((pages * r) // ranks) * PAGE) for r in range(ranks)]
    return b + [seqlen]


@dataclasses.dataclass
class RankSlice:
    """One rank's share of a batch: for request i its tokens
    [start[i], start[i] + length[i]) of the request."""
    start: List[int]
    length: List[int]


class DeviceSteps:
    """The per-rank steps on the GPU through the library's C ABI.

    q_fp8, q_scale, w, q: the batch's (replicated) queries; k_fp8, k_scale,
    kv: this rank's caches; page_table [B, max_pages] int32 and seqlens [B]
    int32 (the slice lengths) describe the rank's local cache; num_pages the
    rows of its caches / 64.
    """

    def __init__(self, q_fp8, q_scale, w, q, k_fp8, k_scale, kv, seqlens, page_table, num_pages,
                 topk, num_heads, sm_scale):
        self.q_fp8, self.q_scale, self.w, self.q = q_fp8, q_scale, w, q
        self.k_fp8, self.k_scale, self.kv = k_fp8, k_scale, kv
        self.seqlens, self.page_table = seqlens, page_table
        self.num_pages, self.topk, self.num_heads = int(num_pages), int(topk), int(num_heads)
        self.sm_scale = float(sm_scale)
        self.dev = q.device
        self.desc = api.make_desc(seqlens, page_table, 1, num_heads, topk, num_pages)
        self.ld = int(page_table.shape[1]) * PAGE

    def scores(self) -> torch.Tensor:
        T = int(self.seqlens.shape[0])
        logits = torch.full((T, self.ld), float("-inf"), dtype=torch.float32, device=self.dev)
        api.dsa_indexer_logits(self.desc, self.q_fp8, self.q_scale, self.w, self.k_fp8,
                               self.k_scale, logits, self.ld)
        return logits

    def local_topk(self, logits: torch.Tensor) -> torch.Tensor:
        T = int(logits.shape[0])
        out = torch.empty((T, self.topk), dtype=torch.int32, device=self.dev)
        ws = torch.empty(api.dsa_topk_workspace_bytes(self.desc, self.ld), dtype=torch.uint8,
                         device=self.dev)
        api.dsa_topk(self.desc, logits, out, ws, self.ld)
        return out

    def global_topk(self, cand_scores: torch.Tensor) -> torch.Tensor:
        """Top-k over the rows of cand_scores [T, n] (n = R * k candidates,
        -inf for padding): indices into the row, ascending, -1 padded."""
        T, n = (int(x) for x in cand_scores.shape)
        seq = torch.full((T,), n, dtype=torch.int32, device=self.dev)
        table = torch.zeros((T, n // PAGE), dtype=torch.int32, device=self.dev)
        desc = api.make_desc(seq, table, 1, self.num_heads, self.topk, n // PAGE)
        out = torch.empty((T, self.topk), dtype=torch.int32, device=self.dev)
        ws = torch.empty(api.dsa_topk_workspace_bytes(desc, n), dtype=torch.uint8, device=self.dev)
        api.dsa_topk(desc, cand_scores.contiguous(), out, ws, n)
        return out

    def attention(self, idx_local: torch.Tensor):
        T, H = int(idx_local.shape[0]), self.num_heads
        mid_o = torch.empty((T, H, 1, 512), dtype=torch.float32, device=self.dev)
        mid_lse = torch.empty((T, H, 1), dtype=torch.float32, device=self.dev)
        api.dsa_sparse_mla_decode_split(self.desc, self.q, self.kv, idx_local.contiguous(), 1,
                                        self.sm_scale, mid_o, mid_lse)
        return mid_o.view(T, H, 512), mid_lse.view(T, H)

    def merge(self, mid_o: torch.Tensor, mid_lse: torch.Tensor) -> torch.Tensor:
        T, H, R, _ = (int(x) for x in mid_o.shape)
        out = torch.empty((T, H, 512), dtype=torch.float32, device=self.dev)
        api.dsa_merge(T * H, R, mid_o.contiguous(), mid_lse.contiguous(), out)
        return out


def phase_a(steps, sl: RankSlice):
    """Local scores and top-k: (candidate scores [T, k] float32, -inf where
    none; their global positions [T, k] int32, -1 where none)."""
    logits = steps.scores()
    loc = steps.local_topk(logits).long()
    valid = loc >= 0
    sc = torch.gather(logits, 1, loc.clamp(min=0))
    sc = torch.where(valid, sc, torch.full_like(sc, float("-inf")))
    start = torch.tensor(sl.start, dtype=torch.long, device=loc.device).view(-1, 1)
    pos = torch.where(valid, loc + start, torch.full_like(loc, -1))
    return sc.float().contiguous(), pos.int().contiguous()


def phase_b(steps, sl: RankSlice, cand_scores: torch.Tensor, cand_pos: torch.Tensor):
    """The global winners from all ranks' candidates ([T, R * k] each, rank-
    major), then the attention over those this rank holds."""
    sel = steps.global_topk(cand_scores).long()
    gpos = torch.gather(cand_pos.long(), 1, sel.clamp(min=0))
    gpos = torch.where(sel >= 0, gpos, torch.full_like(gpos, -1))
    start = torch.tensor(sl.start, dtype=torch.long, device=gpos.device).view(-1, 1)
    length = torch.tensor(sl.length, dtype=torch.long, device=gpos.device).view(-1, 1)
    own = (gpos >= start) & (gpos < start + length)
    # This rank's winners, moved to the front of the row in ascending order
    # (the attention reads the first min(k, slice length) entries), -1 after.
    order = torch.argsort((~own).to(torch.int8), dim=1, stable=True)
    local = torch.where(own, gpos - start, torch.full_like(gpos, -1))
    idx_local = torch.gather(local, 1, order).int()
    mid_o, mid_lse = steps.attention(idx_local)
    # The selection as positions, ascending, -1 after (padding candidates are
    # chosen only when fewer than k exist, and may sit between valid ones).
    sel_pos = torch.gather(gpos, 1, torch.argsort((gpos < 0).to(torch.int8), dim=1, stable=True))
    return mid_o, mid_lse, sel_pos.int()


def _stack_ranks(parts: Sequence[torch.Tensor], dim: int) -> torch.Tensor:
    return torch.stack(list(parts), dim=dim).contiguous()


def run_distributed(steps, sl: RankSlice, group=None):
    """One context-parallel decode layer on this rank of `group` (every rank
    calls it with its own steps and slice).  Returns (out [T, H, 512], the
    global selection as positions [T, k] int32, -1 padded) on every rank."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    sc, pos = phase_a(steps, sl)
    sc_all = [torch.empty_like(sc) for _ in range(R)]
    pos_all = [torch.empty_like(pos) for _ in range(R)]
    dist.all_gather(sc_all, sc, group=group)
    dist.all_gather(pos_all, pos, group=group)
    mid_o, mid_lse, sel = phase_b(steps, sl, torch.cat(sc_all, 1), torch.cat(pos_all, 1))
    o_all = [torch.empty_like(mid_o) for _ in range(R)]
    l_all = [torch.empty_like(mid_lse) for _ in range(R)]
    dist.all_gather(o_all, mid_o, group=group)
    dist.all_gather(l_all, mid_lse, group=group)
    out = steps.merge(_stack_ranks(o_all, 2), _stack_ranks(l_all, 2))
    return out, sel


def run_emulated(steps_per_rank: Sequence, slices: Sequence[RankSlice]):
    """The same layer with R ranks emulated one after another in this process
    (each rank's steps on its own caches; the exchanges are concatenations).
    Returns (out, selection) as run_distributed does."""
    a = [phase_a(s, sl) for s, sl in zip(steps_per_rank, slices)]
    cand_scores = torch.cat([x[0] for x in a], 1)
    cand_pos = torch.cat([x[1] for x in a], 1)
    b = [phase_b(s, sl, cand_scores, cand_pos) for s, sl in zip(steps_per_rank, slices)]
    out = steps_per_rank[0].merge(_stack_ranks([x[0] for x in b], 2),
                                  _stack_ranks([x[1] for x in b], 2))
    return out, b[0][2]
