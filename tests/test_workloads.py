"""The synthetic inputs follow their stated recipe (CPU).

Shapes and distributions of the six workloads: request counts, query tokens
per request, context lengths, heads, k; page tables that map every request's
pages to distinct physical pages; heavy tokens planted uniformly or in
contiguous runs; per-token FP8 scales; the second layer's keys close to the
first's.
"""
import numpy as np
import pytest
import torch

from deepseek_sparse_attention_lightning_gb300 import workloads as W


def test_specs_match_the_workload_table():
    S = W.SPECS
    assert (S["tiny_4k"].batch, S["tiny_4k"].q_per_req, S["tiny_4k"].num_heads,
            S["tiny_4k"].seqlen, S["tiny_4k"].paged) == (1, 1, 16, 4096, False)
    assert (S["mtp_32k"].batch, S["mtp_32k"].q_per_req, S["mtp_32k"].seqlen) == (32, 2, 32769)
    assert (S["long_varlen"].batch, S["long_varlen"].seqlen) == (8, (65536, 131072))
    assert (S["long_128k"].batch, S["long_128k"].seqlen) == (8, 131072)
    assert (S["short_dense"].batch, S["short_dense"].seqlen) == (128, (512, 2048))
    assert (S["mli_195k"].batch, S["mli_195k"].seqlen, S["mli_195k"].layers) == (4, 196608, 2)
    for name, spec in S.items():
        assert spec.topk == 2048
        assert spec.num_heads == (16 if name == "tiny_4k" else 128)
        assert spec.sm_scale == pytest.approx(1 / np.sqrt(192))


@pytest.mark.parametrize("paged", [True, False])
def test_page_tables_map_requests_to_distinct_pages(paged):
    spec = W.small_spec("long_varlen", batch=5, seed=9, paged=paged)
    wl = W.make_workload(spec, seqlens=[64, 65, 1000, 1, 4096])
    table = wl.page_table.numpy()
    used = []
    for r, s in enumerate(wl.seqlens.tolist()):
        n = -(-s // 64)
        assert (table[r, :n] >= 0).all() and (table[r, :n] < wl.num_pages).all()
        assert (table[r, n:] == -1).all()
        used.extend(table[r, :n].tolist())
    assert len(used) == len(set(used)) == wl.num_pages
    if not paged:
        assert used == list(range(wl.num_pages))


def test_variable_lengths_stay_in_their_range():
    spec = W.small_spec("short_dense", batch=64, seed=3)
    s = W.make_workload(spec).seqlens.numpy()
    lo, hi = spec.seqlen
    assert (s >= lo).all() and (s <= hi).all() and len(set(s.tolist())) > 1


def test_heavy_tokens_in_contiguous_runs():
    rng = np.random.default_rng(0)
    pos = W._heavy_positions(rng, "runs:0.005:8", 131072)
    assert abs(len(pos) - round(0.005 * 131072)) <= 8
    breaks = np.flatnonzero(np.diff(pos) > 1)
    assert len(breaks) + 1 <= 8                    # at most 8 runs (adjacent runs may touch)
    uni = W._heavy_positions(np.random.default_rng(0), "frac:0.01", 32769)
    assert len(uni) == round(0.01 * 32769) and len(np.unique(uni)) == len(uni)


def test_fp8_scales_and_second_layer_keys():
    spec = W.small_spec("mli_195k", batch=2, seed=4)
    wl = W.make_workload(spec, seqlens=[700, 900])
    for lc in wl.layers:
        assert (lc.k_scale > 0).all()
        codes = lc.k_fp8.view(torch.float8_e4m3fn).float()
        # amax/448 scales: every token's largest code is +-448
        assert torch.allclose(codes.abs().amax(dim=1), torch.full((codes.shape[0],), 448.0))
    k1 = wl.layers[0].k_fp8.view(torch.float8_e4m3fn).float() * wl.layers[0].k_scale[:, None]
    k2 = wl.layers[1].k_fp8.view(torch.float8_e4m3fn).float() * wl.layers[1].k_scale[:, None]
    # layer-2 keys are layer-1 keys plus N(0, 0.2) noise
    d = (k2 - k1).flatten()
    assert 0.15 < float(d.std()) < 0.25
    assert float(torch.corrcoef(torch.stack([k1.flatten(), k2.flatten()]))[0, 1]) > 0.95


def test_mtp_queries_share_few_selections():
    """The two query tokens of an mtp_32k request draw independent index
    queries, so their selections overlap little (the heavy tokens and
    chance): the oracle's selections of four requests share < 10 % of their
    positions, i.e. a gather of the union would read > 90 % of 2k rows."""
    import numpy as np
    import oracle as O
    from deepseek_sparse_attention_lightning_gb300 import workloads as W
    a = W.host_arrays(W.make_workload("mtp_32k"))
    nq, k = a["q_per_req"], a["topk"]
    shared = []
    for r in range(4):
        sl = slice(r * nq, (r + 1) * nq)
        I, _ = O.indexer_logits(a["q_fp8"][sl], a["q_scale"][sl], a["w"][sl], a["k_fp8"],
                                a["k_scale"], a["page_table"][r:r + 1], a["seqlens"][r:r + 1], nq,
                                with_bound=False)
        sel = O.topk(I.astype(np.float32), O.visible_lengths(a["seqlens"][r:r + 1], nq), k)
        assert (sel >= 0).sum(axis=1).tolist() == [k, k]
        shared.append(len(set(sel[0].tolist()) & set(sel[1].tolist())))
    assert 0 < np.mean(shared) < 0.1 * k
