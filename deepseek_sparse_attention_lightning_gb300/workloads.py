"""Seeded synthetic DSA decode workloads.

This module draws random inputs and lays them out in the cache format the
library consumes.  It holds none of the method's arithmetic: no scoring, no
selection, no softmax, no visibility rule.  Both the float64 oracle (under
``oracle/``) and the CUDA path read the bytes produced here, so it is the one
piece of code the two sides share.

Recipe (shapes and distributions of the workloads on the pages):

* Lightning-indexer queries ``q^I`` [T, 64, 128] and keys ``k^I`` [rows, 128]
  are drawn N(0, 1), then cast to FP8 E4M3 with one fp32 scale per token,
  ``scale = amax / 448`` (amax over all 64x128 query values of a query token,
  over the 128 values of a key token).  Head weights ``w`` [T, 64] ~ N(0,1)/8.
  ("MTP and sparse attention: NSA and DSA", section "Sparse attention: NSA and
  DSA": 64 indexer heads of 128 dims in FP8, one 4-byte scale per cached key.)
* MLA queries [T, H, 576] and the latent cache [rows, 576] (kv_lora_rank 512 +
  rope 64) are bf16 N(0, 1).
* "Heavy" tokens: the index key of a planted token is set to the first query
  token's index query for its highest-weighted head, plus N(0, 0.1) noise,
  before FP8 quantisation, so that it scores high.
* Caches are paged with 64 tokens per page.  The page table maps each
  request's logical page to a physical page; a random permutation of the
  physical pages (or the identity for a contiguous cache).  Table entries past
  a request's last page hold -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

INDEX_HEADS = 64
INDEX_DIM = 128
LATENT_DIM = 576          # kv_lora_rank 512 + qk_rope_head_dim 64
V_DIM = 512
PAGE_SIZE = 64
FP8_E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and distribution of one synthetic decode batch.

    seqlen: cached tokens per request *including* the request's new query
    tokens; an int (fixed) or an inclusive (lo, hi) range drawn uniformly.
    heavy: 'none', 'count:N' (N uniform positions), 'frac:F' (F*S uniform
    positions) or 'runs:F:R' (F*S positions in R contiguous runs).
    """
    name: str
    batch: int
    q_per_req: int
    num_heads: int
    topk: int
    seqlen: object
    heavy: str = "none"
    paged: bool = True
    layers: int = 1
    layer2_noise: float = 0.0
    sm_scale: float = 1.0 / math.sqrt(192.0)
    seed: int = 0
    spare_pages: int = 0

    @property
    def num_tokens(self) -> int:
        return self.batch * self.q_per_req


# The five workloads of the benchmark, plus the fixed-128K variant of the long
# variable-length decode on which the headline figure is quoted.
SPECS = {
    "tiny_4k": WorkloadSpec("tiny_4k", batch=1, q_per_req=1, num_heads=16, topk=2048,
                            seqlen=4096, heavy="count:64", paged=False, seed=0),
    "mtp_32k": WorkloadSpec("mtp_32k", batch=32, q_per_req=2, num_heads=128, topk=2048,
                            seqlen=32769, heavy="frac:0.01", paged=True, seed=1),
    "long_varlen": WorkloadSpec("long_varlen", batch=8, q_per_req=1, num_heads=128, topk=2048,
                                seqlen=(65536, 131072), heavy="runs:0.005:8", paged=True, seed=2),
    "long_128k": WorkloadSpec("long_128k", batch=8, q_per_req=1, num_heads=128, topk=2048,
                              seqlen=131072, heavy="runs:0.005:8", paged=True, seed=2),
    "short_dense": WorkloadSpec("short_dense", batch=128, q_per_req=1, num_heads=128, topk=2048,
                                seqlen=(512, 2048), heavy="none", paged=True, seed=3),
    "mli_195k": WorkloadSpec("mli_195k", batch=4, q_per_req=1, num_heads=128, topk=2048,
                             seqlen=196608, heavy="runs:0.005:8", paged=True, layers=2,
                             layer2_noise=0.2, seed=4),
}


@dataclasses.dataclass
class LayerCache:
    """Per-layer tensors: the two caches and the MLA query."""
    k_fp8: torch.Tensor      # uint8 [rows, 128]   FP8 E4M3 bytes
    k_scale: torch.Tensor    # float32 [rows]
    q: torch.Tensor          # bfloat16 [T, H, 576]
    kv: torch.Tensor         # bfloat16 [rows, 576]


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seqlens: torch.Tensor    # int32 [B]
    page_table: torch.Tensor  # int32 [B, max_pages]
    num_pages: int
    q_fp8: torch.Tensor      # uint8 [T, 64, 128]
    q_scale: torch.Tensor    # float32 [T]
    w: torch.Tensor          # float32 [T, 64]
    layers: list             # list[LayerCache]
    heavy: list              # per request: np.ndarray of logical positions

    # convenience accessors for layer 0
    @property
    def k_fp8(self):
        return self.layers[0].k_fp8

    @property
    def k_scale(self):
        return self.layers[0].k_scale

    @property
    def q(self):
        return self.layers[0].q

    @property
    def kv(self):
        return self.layers[0].kv

    def to(self, device) -> "Workload":
        """A copy with every tensor moved to ``device`` (same bytes)."""
        mv = lambda t: t.to(device)
        return Workload(spec=self.spec, seqlens=mv(self.seqlens), page_table=mv(self.page_table),
                        num_pages=self.num_pages, q_fp8=mv(self.q_fp8), q_scale=mv(self.q_scale),
                        w=mv(self.w),
                        layers=[LayerCache(k_fp8=mv(l.k_fp8), k_scale=mv(l.k_scale), q=mv(l.q),
                                           kv=mv(l.kv)) for l in self.layers],
                        heavy=self.heavy)

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_seqlen(self) -> int:
        return int(self.seqlens.max().item())


def _quantize_rows_e4m3(x: torch.Tensor, rows_dim_start: int):
    """Cast ``x`` to FP8 E4M3 with one scale per leading index (amax/448).

    Returns (uint8 bytes, float32 scales).  Scaling and the cast are input
    preparation (the pages store FP8 keys with a per-token scale); the cast
    itself is torch's round-to-nearest conversion.
    """
    flat = x.reshape(x.shape[0], -1).float()
    amax = flat.abs().amax(dim=1).clamp_min(1e-12)
    scale = (amax / FP8_E4M3_MAX).float()
    y = (flat / scale[:, None]).clamp(-FP8_E4M3_MAX, FP8_E4M3_MAX)
    q8 = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(x.shape)
    return q8.contiguous(), scale.contiguous()


def _heavy_positions(rng: np.random.Generator, mode: str, s: int) -> np.ndarray:
    if mode == "none" or s <= 0:
        return np.zeros(0, dtype=np.int64)
    kind, *args = mode.split(":")
    if kind == "count":
        n = min(int(args[0]), s)
        return np.sort(rng.choice(s, size=n, replace=False))
    if kind == "frac":
        n = min(max(1, int(round(float(args[0]) * s))), s)
        return np.sort(rng.choice(s, size=n, replace=False))
    if kind == "runs":
        frac, runs = float(args[0]), int(args[1])
        total = max(runs, int(round(frac * s)))
        run_len = max(1, total // runs)
        seg = s // runs
        out = []
        for i in range(runs):
            lo = i * seg
            span = max(1, seg - run_len)
            start = lo + int(rng.integers(0, span))
            out.append(np.arange(start, min(start + run_len, s)))
        return np.unique(np.concatenate(out))
    raise ValueError(f"unknown heavy mode {mode!r}")


def make_workload(spec: WorkloadSpec | str, device: str | torch.device = "cpu",
                  seqlens: Optional[list] = None) -> Workload:
    """Draw the workload described by ``spec`` (seeded by ``spec.seed``).

    Integers (sequence lengths, page permutation, heavy positions) come from a
    numpy generator and are identical on every device; the float arrays come
    from a torch generator on ``device``.
    """
    if isinstance(spec, str):
        spec = SPECS[spec]
    device = torch.device(device)
    rng = np.random.default_rng(spec.seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)

    B, nq, H = spec.batch, spec.q_per_req, spec.num_heads
    T = B * nq
    if seqlens is not None:
        s_arr = np.asarray(seqlens, dtype=np.int64)
    elif isinstance(spec.seqlen, (tuple, list)):
        lo, hi = spec.seqlen
        s_arr = rng.integers(lo, hi + 1, size=B)
    else:
        s_arr = np.full(B, int(spec.seqlen), dtype=np.int64)
    assert s_arr.shape == (B,)
    pages_per_req = [(int(s) + PAGE_SIZE - 1) // PAGE_SIZE for s in s_arr]
    used_pages = int(sum(pages_per_req))
    num_pages = used_pages + spec.spare_pages
    max_pages = max(1, max(pages_per_req))
    phys = rng.permutation(num_pages) if spec.paged else np.arange(num_pages)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(pages_per_req):
        table[r, :n] = phys[off:off + n]
        off += n
    rows = num_pages * PAGE_SIZE

    def randn(*shape, dtype=torch.float32):
        return torch.randn(*shape, generator=gen, device=device, dtype=dtype)

    q_idx = randn(T, INDEX_HEADS, INDEX_DIM)
    w = (randn(T, INDEX_HEADS) / 8.0).contiguous()
    k_idx = randn(rows, INDEX_DIM)

    heavy = [_heavy_positions(rng, spec.heavy, int(s)) for s in s_arr]
    table_t = torch.from_numpy(table)
    for r in range(B):
        pos = heavy[r]
        if pos.size == 0:
            continue
        t0 = r * nq
        j_star = int(torch.argmax(w[t0]).item())
        pos_t = torch.from_numpy(pos)
        prow = (table_t[r, pos_t // PAGE_SIZE].long() * PAGE_SIZE + pos_t % PAGE_SIZE).to(device)
        noise = randn(pos.size, INDEX_DIM) * 0.1
        k_idx[prow] = q_idx[t0, j_star][None, :] + noise

    q_fp8, q_scale = _quantize_rows_e4m3(q_idx, 1)
    k_fp8, k_scale = _quantize_rows_e4m3(k_idx, 1)
    layers = [LayerCache(k_fp8=k_fp8, k_scale=k_scale,
                         q=randn(T, H, LATENT_DIM, dtype=torch.bfloat16),
                         kv=randn(rows, LATENT_DIM, dtype=torch.bfloat16))]
    for _ in range(1, spec.layers):
        k2 = k_idx + spec.layer2_noise * randn(rows, INDEX_DIM)
        k2_fp8, k2_scale = _quantize_rows_e4m3(k2, 1)
        layers.append(LayerCache(k_fp8=k2_fp8, k_scale=k2_scale,
                                 q=randn(T, H, LATENT_DIM, dtype=torch.bfloat16),
                                 kv=randn(rows, LATENT_DIM, dtype=torch.bfloat16)))
        del k2
    del k_idx, q_idx
    return Workload(spec=spec,
                    seqlens=torch.from_numpy(s_arr.astype(np.int32)).to(device),
                    page_table=table_t.to(device),
                    num_pages=num_pages,
                    q_fp8=q_fp8, q_scale=q_scale, w=w, layers=layers, heavy=heavy)


def small_spec(base: str, **overrides) -> WorkloadSpec:
    """A reduced copy of one of the named workloads (for parity tests)."""
    return dataclasses.replace(SPECS[base], **overrides)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_arrays(wl: Workload, layer: int = 0) -> dict:
    """Host numpy copies of every input of one layer, as raw bytes/bits."""
    lc = wl.layers[layer]
    return dict(
        seqlens=wl.seqlens.cpu().numpy().astype(np.int64),
        page_table=wl.page_table.cpu().numpy().astype(np.int64),
        q_per_req=wl.spec.q_per_req,
        q_fp8=wl.q_fp8.cpu().numpy(),
        q_scale=wl.q_scale.cpu().numpy(),
        w=wl.w.cpu().numpy(),
        k_fp8=lc.k_fp8.cpu().numpy(),
        k_scale=lc.k_scale.cpu().numpy(),
        q=bf16_bits(lc.q),
        kv=bf16_bits(lc.kv),
        sm_scale=wl.spec.sm_scale,
        topk=wl.spec.topk,
    )
