"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (from the stated targets):
  * indexer scores: |gpu - oracle| <= 1e-3 * E, E = sum of |terms| of the score;
  * top-k: bit-exact as a set (and, by the ABI, as a sorted list) when both
    sides select from the same fp32 score tensor;
  * attention (Mid_O, Mid_LSE, merged output): |gpu - oracle| <= 2e-2 + 1e-2 |oracle|
    given identical indices.
Small cases span several tiles and a ragged tail; the workload-sized cases at
the bottom check sampled outputs in the launch configuration the benchmark
times.
"""
import numpy as np
import pytest
import torch

import oracle as O
from deepseek_sparse_attention_lightning_gb300 import api
from deepseek_sparse_attention_lightning_gb300 import workloads as W

pytestmark = pytest.mark.gpu

IDX_REL = 1e-3
ATT_ATOL, ATT_RTOL = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_sparse_attention_lightning_gb300 import build
    build.build()
    api.lib()
    yield
    torch.cuda.synchronize()


def _assert_no_device_error():
    code = api.dsa_get_device_error()
    assert code == 0, api.STATUS_NAMES.get(code, code)


def _gpu_wl(base, seqlens=None, **kw):
    wl = W.make_workload(W.small_spec(base, **kw), seqlens=seqlens)
    return wl, wl.to("cuda")


def _assert_close_att(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(want)
    g, w = np.where(both_inf, 0.0, got), np.where(both_inf, 0.0, want)
    bad = ~(np.abs(g - w) <= ATT_ATOL + ATT_RTOL * np.abs(w))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; " \
                          f"max err {np.nanmax(np.abs(g - w))}"


# ---------------------------------------------------------------- indexer

INDEXER_CASES = [
    dict(base="long_varlen", batch=3, q_per_req=1, seqlens=[130, 700, 257], paged=True, seed=21),
    dict(base="mtp_32k", batch=2, q_per_req=2, seqlens=[300, 901], paged=True, seed=22),
    dict(base="mtp_32k", batch=2, q_per_req=3, seqlens=[200, 450], paged=True, seed=23),
    dict(base="mtp_32k", batch=2, q_per_req=4, seqlens=[129, 384], paged=True, seed=24),
    dict(base="tiny_4k", batch=1, q_per_req=1, seqlens=[4096], paged=False, seed=0),
    dict(base="long_varlen", batch=5, q_per_req=1, seqlens=[1, 64, 65, 127, 1000], paged=True, seed=25),
]


@pytest.mark.parametrize("case", INDEXER_CASES, ids=lambda c: f"{c['base']}-nq{c['q_per_req']}")
def test_indexer_matches_oracle(case):
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, heavy="none", **case)
    logits = api.run_indexer(g).cpu().numpy()
    _assert_no_device_error()
    a = W.host_arrays(wl)
    I, E = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                            a["page_table"], a["seqlens"], a["q_per_req"])
    vis = O.visible_lengths(a["seqlens"], a["q_per_req"])
    nq = a["q_per_req"]
    for t, n in enumerate(vis):
        err = np.abs(logits[t, :n].astype(np.float64) - I[t, :n])
        assert (err <= IDX_REL * E[t, :n] + 1e-30).all(), f"row {t}: max rel {np.max(err / (E[t, :n] + 1e-30))}"
        S = int(a["seqlens"][t // nq])
        tail_end = min(((S + 127) // 128) * 128, logits.shape[1])
        assert np.isneginf(logits[t, n:tail_end]).all()


def test_indexer_head_permutation_invariance_on_gpu():
    wl, g = _gpu_wl("mtp_32k", batch=2, q_per_req=2, seqlens=[500, 700], heavy="none", seed=31)
    l1 = api.run_indexer(g)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(0)).cuda()
    g.q_fp8 = g.q_fp8[:, perm].contiguous()
    g.w = g.w[:, perm].contiguous()
    l2 = api.run_indexer(g)
    vis = O.visible_lengths(wl.seqlens.numpy(), 2)
    for t, n in enumerate(vis):
        a, b = l1[t, :n].cpu().numpy(), l2[t, :n].cpu().numpy()
        assert np.allclose(a, b, rtol=1e-5, atol=1e-4 * np.abs(a).max())


# ---------------------------------------------------------------- top-k

def _topk_desc(vis_rows, ld, k, nq=1):
    """A descriptor whose rows see exactly ``vis_rows`` tokens (nq = 1)."""
    B = len(vis_rows)
    seqlens = torch.tensor(vis_rows, dtype=torch.int32, device="cuda")
    max_pages = ld // 64
    table = torch.zeros((B, max_pages), dtype=torch.int32, device="cuda")
    desc = api.make_desc(seqlens, table, nq, 128, k, max_pages)
    return desc, (seqlens, table)


def _gpu_topk(scores_np, vis_rows, k):
    T, ld = scores_np.shape
    desc, keep = _topk_desc(vis_rows, ld, k)
    logits = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).cuda()
    ws = torch.empty(api.dsa_topk_workspace_bytes(desc, ld), dtype=torch.uint8, device="cuda")
    out = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    api.dsa_topk(desc, logits, out, ws, ld)
    res = out.cpu().numpy()
    _assert_no_device_error()
    return res


TOPK_CASES = {
    # name: (rows, ld, k, generator)
    "gauss_k2048": (4, 20480, 2048, lambda r, n: r.standard_normal(n)),
    "ties_k64": (3, 3072, 64, lambda r, n: np.round(r.standard_normal(n) * 4) / 4),
    "ties_k2048": (3, 9216, 2048, lambda r, n: np.round(r.standard_normal(n) * 2) / 2),
    "all_equal": (2, 8192, 100, lambda r, n: np.zeros(n)),
    "signed_zero": (2, 4096, 300, lambda r, n: np.where(r.random(n) < 0.5, -0.0, 0.0)),
    "heavy_tail": (2, 65536, 2048, lambda r, n: r.standard_normal(n) ** 3),
    "k1": (2, 4096, 1, lambda r, n: r.standard_normal(n)),
}


@pytest.mark.parametrize("name", sorted(TOPK_CASES))
def test_topk_bit_exact(name):
    rows, ld, k, gen = TOPK_CASES[name]
    rng = np.random.default_rng(abs(hash(name)) % 2 ** 31)
    scores = np.stack([gen(rng, ld) for _ in range(rows)]).astype(np.float32)
    vis = [ld - 7 * i for i in range(rows)]
    got = _gpu_topk(scores, vis, k)
    want = O.topk(scores, np.array(vis), k)
    assert np.array_equal(got, want)


def test_topk_short_rows_select_everything():
    rng = np.random.default_rng(1)
    scores = rng.standard_normal((4, 4096)).astype(np.float32)
    vis = [1, 2047, 2048, 2049]
    got = _gpu_topk(scores, vis, 2048)
    want = O.topk(scores, np.array(vis), 2048)
    assert np.array_equal(got, want)
    assert got[0, 0] == 0 and (got[0, 1:] == -1).all()


def test_topk_long_rows():
    rng = np.random.default_rng(2)
    ld = 196608
    scores = rng.standard_normal((3, ld)).astype(np.float32)
    vis = [ld, 131072, 100000]
    got = _gpu_topk(scores, vis, 2048)
    assert np.array_equal(got, O.topk(scores, np.array(vis), 2048))


# ---------------------------------------------------------------- sparse MLA

def _oracle_indices(wl, k=None):
    a = W.host_arrays(wl)
    I, _ = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                            a["page_table"], a["seqlens"], a["q_per_req"], with_bound=False)
    vis = O.visible_lengths(a["seqlens"], a["q_per_req"])
    return a, O.topk(I.astype(np.float32), vis, a["topk"] if k is None else k)


MLA_CASES = [
    dict(base="mtp_32k", batch=2, q_per_req=2, num_heads=128, topk=2048, seqlens=[2600, 3100], seed=41),
    dict(base="tiny_4k", batch=1, q_per_req=1, num_heads=16, topk=2048, seqlens=[4096], seed=0),
    dict(base="short_dense", batch=3, q_per_req=1, num_heads=128, topk=2048, seqlens=[700, 1500, 63], seed=42),
    dict(base="long_varlen", batch=2, q_per_req=1, num_heads=64, topk=256, seqlens=[1000, 333], seed=43),
    dict(base="mtp_32k", batch=1, q_per_req=2, num_heads=48, topk=200, seqlens=[2], seed=44),
]


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("case", MLA_CASES, ids=lambda c: f"{c['base']}-H{c['num_heads']}-k{c['topk']}")
def test_sparse_mla_split_and_merge_match_oracle(case, splits):
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, heavy="none", **case)
    a, idx = _oracle_indices(wl)
    idx_gpu = torch.from_numpy(idx.astype(np.int32)).cuda()
    mid_o, mid_lse = api.run_sparse_mla_split(g, idx_gpu, num_splits=splits)
    S = mid_o.shape[2]
    out, lse = api.run_merge(mid_o, mid_lse)
    _assert_no_device_error()
    mo, ml = O.sparse_mla_split(a["q"], a["kv"], idx, a["page_table"], a["seqlens"],
                                a["q_per_req"], a["sm_scale"], S)
    _assert_close_att(mid_o.cpu().numpy(), mo, "Mid_O")
    _assert_close_att(mid_lse.cpu().numpy(), ml, "Mid_LSE")
    o, l = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], a["q_per_req"],
                        a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")
    _assert_close_att(lse.cpu().numpy(), l, "LSE")


def test_sparse_mla_rows_of_mixed_lengths_in_a_multi_wave_grid():
    """160 rows of 1 to 2048 selected keys, one split: 320 CTAs, more than
    the GPU has SMs, so the CTAs take the rows longest first (the kernel
    ranks them by their selected count).  Every row's Mid_O / LSE must still
    land in its own place: element-wise against the oracle."""
    B = 160
    rng = np.random.default_rng(46)
    lens = rng.integers(1, 2049, size=B)
    lens[:3] = [1, 2048, 64]                              # the extremes and one full tile
    wl, g = _gpu_wl("short_dense", batch=B, q_per_req=1, num_heads=16, topk=2048,
                    seqlens=lens.tolist(), heavy="none", seed=47)
    a = W.host_arrays(wl)
    idx = np.full((B, 2048), -1, dtype=np.int64)
    for t, n in enumerate(lens):
        idx[t, :n] = np.arange(n)
    mid_o, mid_lse = api.run_sparse_mla_split(g, torch.from_numpy(idx.astype(np.int32)).cuda(), 1)
    _assert_no_device_error()
    mo, ml = O.sparse_mla_split(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 1,
                                a["sm_scale"], 1)
    _assert_close_att(mid_o.cpu().numpy(), mo, "Mid_O")
    _assert_close_att(mid_lse.cpu().numpy(), ml, "Mid_LSE")


def test_sparse_mla_skips_padding_and_many_empty_splits():
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[100, 70], heavy="none", seed=45)
    a = W.host_arrays(wl)
    idx = np.full((2, 2048), -1, dtype=np.int64)
    idx[0, :100] = np.random.default_rng(0).permutation(100)
    idx[1, :70] = np.arange(70)
    idx[1, 10] = -1                                     # a hole inside the valid prefix
    mid_o, mid_lse = api.run_sparse_mla_split(g, torch.from_numpy(idx.astype(np.int32)).cuda(), 32)
    out, lse = api.run_merge(mid_o, mid_lse)
    _assert_no_device_error()
    assert torch.isneginf(mid_lse[:, :, 2:]).all()      # splits past the selection are empty
    o, l = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")
    _assert_close_att(lse.cpu().numpy(), l, "LSE")


# ---------------------------------------------------------------- fused layer

FUSED_CASES = [
    dict(base="mtp_32k", batch=3, q_per_req=2, num_heads=128, topk=2048, seqlens=[5000, 2100, 9000],
         heavy="frac:0.01", seed=51),
    dict(base="long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048, seqlens=[20000, 12345],
         heavy="runs:0.005:8", seed=52),
    dict(base="short_dense", batch=4, q_per_req=1, num_heads=128, topk=2048, seqlens=[512, 2048, 1999, 3000],
         heavy="none", seed=53),
    dict(base="tiny_4k", batch=1, q_per_req=1, num_heads=16, topk=2048, seqlens=[4096], heavy="count:64", seed=0),
]


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: c["base"])
def test_fused_decode_layer(case):
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    T, k = wl.spec.num_tokens, wl.spec.topk
    sel = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    out = api.run_decode(g, topk_out=sel)
    logits = api.run_indexer(g)
    _assert_no_device_error()
    a = W.host_arrays(wl)
    vis = O.visible_lengths(a["seqlens"], a["q_per_req"])
    sel_np = sel.cpu().numpy()
    # (1) the fused selection is exactly the top-k of the kernel's fp32 scores
    lg = logits.cpu().numpy()
    assert np.array_equal(sel_np, O.topk(lg, vis, k))
    # (2) every selected token is a true top-k token up to the score tolerance
    I, E = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                            a["page_table"], a["seqlens"], a["q_per_req"])
    for t, n in enumerate(vis):
        if n <= k:
            continue
        kth = np.sort(I[t, :n])[::-1][k - 1]
        chosen = sel_np[t][sel_np[t] >= 0]
        assert (I[t, chosen] >= kth - 2 * IDX_REL * E[t, chosen]).all()
    # (3) the output is the attention over the selected tokens
    o, _ = O.sparse_mla(a["q"], a["kv"], sel_np, a["page_table"], a["seqlens"], a["q_per_req"],
                        a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")


@pytest.mark.parametrize("case", FUSED_CASES[:2], ids=lambda c: c["base"])
def test_host_step_equals_fused_layer(case):
    # dsa_decode_step_host: the step's inputs packed in one pinned host block,
    # one copy in, the fused layer, one copy out.  Same kernels on the same
    # inputs, so the output must equal dsa_decode_fused's bit for bit; two
    # calls in a row, the second on other queries, check that nothing of the
    # first call's block or output is reused.
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    spec = wl.spec
    B, nq, H, mp = spec.batch, spec.q_per_req, spec.num_heads, g.max_pages
    lay = api.dsa_step_layout_get(B, nq, H, mp)
    host_in = torch.zeros(lay.bytes, dtype=torch.uint8).pin_memory()
    dev_in = torch.empty(lay.bytes, dtype=torch.uint8, device="cuda")
    hv = api.step_views(host_in, lay, B, nq, H, mp)
    desc = api.workload_desc(g)
    ws = api.alloc_workspace(g)
    out = torch.empty((spec.num_tokens, H, 512), dtype=torch.float32, device="cuda")
    host_out = torch.full((spec.num_tokens, H, 512), float("nan")).pin_memory()
    for call in range(2):
        if call == 1:     # new MLA queries for the second step
            g.layers[0].q.copy_(torch.randn(g.layers[0].q.shape, generator=torch.Generator().manual_seed(7))
                                .to(torch.bfloat16))
        for name in ("q_fp8", "q_scale", "w", "seqlens", "page_table"):
            hv[name].copy_(getattr(g, name).cpu())
        hv["q"].copy_(g.layers[0].q.cpu())
        want = api.run_decode(g)
        api.dsa_decode_step_host(desc, host_in, dev_in, g.k_fp8, g.k_scale, g.kv, out, host_out, ws,
                                 g.max_seqlen, spec.sm_scale)
        torch.cuda.synchronize()
        _assert_no_device_error()
        assert torch.equal(host_out, want.cpu()), f"call {call}"
        assert torch.equal(out, want), f"call {call}"


def test_host_step_pipeline_matches_fused_layer():
    # HostStepPipeline: five steps with other MLA queries each, copies on side
    # streams overlapping the neighbouring layers; every step's host output
    # must equal a direct dsa_decode_fused call on the same inputs, bit for bit.
    case = dict(FUSED_CASES[0])
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    spec = wl.spec
    B, nq, H, mp, T = spec.batch, spec.q_per_req, spec.num_heads, g.max_pages, spec.num_tokens
    pipe = api.HostStepPipeline(B, nq, H, spec.topk, mp, g.num_pages, g.max_seqlen, spec.sm_scale)
    lay = pipe.layout
    steps = 5
    qs = [torch.randn(g.q.shape, generator=torch.Generator().manual_seed(100 + i)).to(torch.bfloat16)
          for i in range(steps)]
    host_in, host_out = [], []
    for i in range(steps):
        hb = torch.zeros(lay.bytes, dtype=torch.uint8).pin_memory()
        hv = api.step_views(hb, lay, B, nq, H, mp)
        for name in ("q_fp8", "q_scale", "w", "seqlens", "page_table"):
            hv[name].copy_(getattr(g, name).cpu())
        hv["q"].copy_(qs[i])
        host_in.append(hb)
        host_out.append(torch.full((T, H, 512), float("nan")).pin_memory())
    for i in range(steps):
        pipe.submit(host_in[i], host_out[i], g.k_fp8, g.k_scale, g.kv)
    pipe.drain()
    torch.cuda.synchronize()
    _assert_no_device_error()
    for i in range(steps):
        g.layers[0].q.copy_(qs[i].cuda())
        want = api.run_decode(g)
        torch.cuda.synchronize()
        assert torch.equal(host_out[i], want.cpu()), f"step {i}"


def test_fused_reuses_given_selection_on_second_stream():
    # Multi-layer-indexer schedule: layer 2 attends layer 1's selection while
    # layer 2's own indexer + top-k run on another stream.
    wl, g = _gpu_wl("mli_195k", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[6000, 9000], seed=61)
    T, k = wl.spec.num_tokens, wl.spec.topk
    sel1 = torch.empty((T, k), dtype=torch.int32, device="cuda")
    sel2 = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out1 = api.run_decode(g, layer=0, topk_out=sel1)
    side = torch.cuda.Stream()
    ws2 = api.alloc_workspace(g)
    ev = torch.cuda.Event()
    ev.record()
    side.wait_event(ev)
    out2 = api.run_decode(g, layer=1, topk_in=sel1)           # attention of layer 2 (main)
    with torch.cuda.stream(side):
        logits2 = api.run_indexer(g, layer=1, stream=side)     # indexer of layer 2 (side)
        api.dsa_topk(api.workload_desc(g), logits2, sel2,
                     torch.empty(api.dsa_topk_workspace_bytes(api.workload_desc(g), logits2.shape[1]),
                                 dtype=torch.uint8, device="cuda"), stream=side)
    torch.cuda.synchronize()
    _assert_no_device_error()
    a2 = W.host_arrays(wl, layer=1)
    s1 = sel1.cpu().numpy()
    o2, _ = O.sparse_mla(a2["q"], a2["kv"], s1, a2["page_table"], a2["seqlens"], 1, a2["sm_scale"])
    _assert_close_att(out2.cpu().numpy(), o2, "layer-2 output on layer-1 selection")
    vis = O.visible_lengths(a2["seqlens"], 1)
    assert np.array_equal(sel2.cpu().numpy(), O.topk(logits2.cpu().numpy(), vis, k))
    # adjacent layers select overlapping sets (the premise of the schedule)
    s2 = sel2.cpu().numpy()
    overlap = np.mean([len(np.intersect1d(s1[t], s2[t])) / k for t in range(T)])
    assert overlap > 0.2


@pytest.mark.parametrize("nq,splits", [(1, 0), (2, 0), (1, 1), (1, 3)],
                         ids=["nq1-auto", "nq2-auto", "nq1-s1", "nq1-s3"])
def test_mli_layer_matches_separate_calls(nq, splits):
    # dsa_decode_mli: layer 2's attention over layer 1's selection, with layer
    # 2's indexer + top-k on the SMs the attention leaves free (one stream).
    # Its selection must equal the fused layer's bit for bit, its output the
    # oracle's attention over layer 1's selection.
    wl, g = _gpu_wl("mli_195k", batch=3, q_per_req=nq, num_heads=128, topk=2048,
                    seqlens=[6000, 9000, 2500], seed=62 + nq)
    T, k, H = wl.spec.num_tokens, wl.spec.topk, wl.spec.num_heads
    desc = api.workload_desc(g)
    sel1 = torch.empty((T, k), dtype=torch.int32, device="cuda")
    api.run_decode(g, layer=0, topk_out=sel1)
    sel2_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
    api.run_decode(g, layer=1, topk_out=sel2_ref)
    want = api.run_decode(g, layer=1, topk_in=sel1)
    lc2 = g.layers[1]
    ws = api.alloc_workspace(g, splits)
    out = torch.full((T, H, 512), float("nan"), device="cuda")
    sel2 = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    for _ in range(2):      # twice: the second call starts from the first call's workspace
        api.dsa_decode_mli(desc, g.q_fp8, g.q_scale, g.w, lc2.k_fp8, lc2.k_scale, lc2.q, lc2.kv,
                           sel1, sel2, out, ws, g.max_seqlen, wl.spec.sm_scale, splits)
        torch.cuda.synchronize()
        _assert_no_device_error()
        assert torch.equal(sel2, sel2_ref)
        # another split count rounds P (bf16) under other running maxima
        _assert_close_att(out.cpu().numpy(), want.cpu().numpy(), "MLI vs fused (topk_in)")
    a2 = W.host_arrays(wl, layer=1)
    o2, _ = O.sparse_mla(a2["q"], a2["kv"], sel1.cpu().numpy(), a2["page_table"], a2["seqlens"],
                         nq, a2["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o2, "MLI layer output on layer-1 selection")


# ---------------------------------------------------------------- context parallel

def test_context_parallel_emulated_matches_fused_layer():
    """Three ranks, each holding a page-aligned slice of every request (its
    caches seen through the slice's page table), emulated one after another:
    local scores and top-k, the global top-k over the ranks' candidates, the
    attention over each rank's own winners, the merge of the three partials.
    Scores of a token do not depend on the slice it is scored in, so the
    selection equals the fused layer's bit for bit; the output matches it
    and the oracle within the attention tolerance."""
    from deepseek_sparse_attention_lightning_gb300 import cp
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[9000, 5200], heavy="runs:0.005:8", seed=81)
    spec, lc = wl.spec, g.layers[0]
    T, k, H, R = spec.num_tokens, spec.topk, spec.num_heads, 3
    want_sel = torch.empty((T, k), dtype=torch.int32, device="cuda")
    want = api.run_decode(g, topk_out=want_sel)
    seqlens = g.seqlens.cpu().tolist()
    bounds = [cp.slice_bounds(int(S), R) for S in seqlens]
    steps, slices = [], []
    for r in range(R):
        mine = [(b[r], b[r + 1]) for b in bounds]
        npg = [(hi - lo + 63) // 64 for lo, hi in mine]
        table = torch.full((len(mine), max(npg)), -1, dtype=torch.int32, device="cuda")
        for i, (lo, _) in enumerate(mine):
            table[i, :npg[i]] = g.page_table[i, lo // 64: lo // 64 + npg[i]]
        seq = torch.tensor([hi - lo for lo, hi in mine], dtype=torch.int32, device="cuda")
        steps.append(cp.DeviceSteps(g.q_fp8, g.q_scale, g.w, lc.q, lc.k_fp8, lc.k_scale, lc.kv, seq,
                                    table, g.num_pages, k, H, spec.sm_scale))
        slices.append(cp.RankSlice(start=[lo for lo, _ in mine], length=[hi - lo for lo, hi in mine]))
    out, sel = cp.run_emulated(steps, slices)
    torch.cuda.synchronize()
    _assert_no_device_error()
    assert torch.equal(sel, want_sel)
    _assert_close_att(out.cpu().numpy(), want.cpu().numpy(), "context parallel vs fused layer")
    a = W.host_arrays(wl)
    o, _ = O.sparse_mla(a["q"], a["kv"], sel.cpu().numpy(), a["page_table"], a["seqlens"], 1,
                        a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "context parallel vs oracle")


# ---------------------------------------------------------------- errors

def test_device_check_flags_bad_page_id():
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[3000, 700], heavy="none", seed=71)
    g.page_table[0, 3] = wl.num_pages + 5               # outside the cache
    logits = api.run_indexer(g)
    assert api.dsa_get_device_error() == 5               # DSA_ERR_DEVICE_CHECK
    assert api.dsa_get_device_error() == 0               # read-and-clear
    row = logits[0].cpu().numpy()
    assert np.isneginf(row[3 * 64:4 * 64]).all()         # the bad page's tokens are masked
    assert np.isfinite(row[:3 * 64]).all()


def test_device_check_flags_bad_page_ids_in_both_lookup_paths():
    """One 131072-token request: every CTA of the indexer's grid streams 6-7
    tiles of 128 tokens, its first four looked up by the producer itself and
    the rest from the page ids the other warps stage in shared memory.  An
    out-of-range page id in CTA 0's fifth tile (the staged path) and a
    negative one in CTA 1's second tile (the producer's own lookup) must both
    be reported and mask exactly their 64 tokens."""
    wl, g = _gpu_wl("long_varlen", batch=1, q_per_req=1, num_heads=16, topk=2048,
                    seqlens=[131072], heavy="none", seed=74)
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = 131072 // 128
    assert tiles // ctas >= 5
    page_a = 2 * 4 + 1                       # CTA 0, tile 4, its second page
    page_b = 2 * (tiles // ctas + 1)         # CTA 1, its second tile, first page
    g.page_table[0, page_a] = wl.num_pages + 5
    g.page_table[0, page_b] = -3
    assert api.dsa_get_device_error() == 0
    logits = api.run_indexer(g)
    assert api.dsa_get_device_error() == 5               # DSA_ERR_DEVICE_CHECK
    row = logits[0].cpu().numpy()[:131072]
    bad = np.zeros(131072, dtype=bool)
    for pg in (page_a, page_b):
        bad[pg * 64:(pg + 1) * 64] = True
    assert np.isneginf(row[bad]).all()
    assert np.isfinite(row[~bad]).all()


def test_indexer_wait_timeout_is_reported_and_context_survives():
    """A wait bound of one SM cycle makes the indexer's pipeline waits run out
    (the copies they wait for take microseconds): the call must come back,
    report DSA_ERR_TIMEOUT through dsa_get_device_error, and leave the context
    usable -- the same call with the default bound then matches the oracle."""
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[2500, 900], heavy="none", seed=73)
    assert api.dsa_get_device_error() == 0
    try:
        api.dsa_debug_set_wait_cycles(1)
        api.run_indexer(g)
        assert api.dsa_get_device_error() == 6           # DSA_ERR_TIMEOUT
    finally:
        api.dsa_debug_set_wait_cycles(0)
    assert api.dsa_get_device_error() == 0               # read-and-clear
    logits = api.run_indexer(g).cpu().numpy()
    _assert_no_device_error()
    a = W.host_arrays(wl)
    I, E = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                            a["page_table"], a["seqlens"], a["q_per_req"])
    for t, n in enumerate(O.visible_lengths(a["seqlens"], a["q_per_req"])):
        assert (np.abs(logits[t, :n] - I[t, :n]) <= IDX_REL * E[t, :n] + 1e-30).all()


def test_fused_layer_wait_timeout_is_reported_and_context_survives():
    """The fused layer with the indexer's waits bounded by one SM cycle: the
    call comes back with DSA_ERR_TIMEOUT, and the next call with the default
    bound selects exactly and attends correctly (the context stays usable)."""
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=32, topk=2048,
                    seqlens=[9000, 5000], heavy="none", seed=74)
    T, k = wl.spec.num_tokens, wl.spec.topk
    assert api.dsa_get_device_error() == 0
    try:
        api.dsa_debug_set_wait_cycles(1)
        api.run_decode(g)
        assert api.dsa_get_device_error() == 6           # DSA_ERR_TIMEOUT
    finally:
        api.dsa_debug_set_wait_cycles(0)
    sel = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    out = api.run_decode(g, topk_out=sel)
    logits = api.run_indexer(g)
    _assert_no_device_error()
    a = W.host_arrays(wl)
    vis = O.visible_lengths(a["seqlens"], 1)
    sel_np = sel.cpu().numpy()
    assert np.array_equal(sel_np, O.topk(logits.cpu().numpy(), vis, k))
    o, _ = O.sparse_mla(a["q"], a["kv"], sel_np, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O after a timed-out call")


# ---------------------------------------------------------------- fused selection

# The fused layer's selection (the indexer's histogram, then the top-k) must
# be the top-k of the same scores bit for bit, across query counts, k, row
# lengths and batch sizes.
SEL_CASES = [
    # n_q = 3: rows at, just above and far above k, several requests
    dict(base="mtp_32k", batch=4, q_per_req=3, num_heads=16, topk=2048,
         seqlens=[2049, 7000, 2050, 15000], heavy="frac:0.01", seed=81),
    # n_q = 4
    dict(base="mtp_32k", batch=3, q_per_req=4, num_heads=32, topk=2048,
         seqlens=[9000, 2051, 4100], heavy="frac:0.01", seed=82),
    # n_q = 2: a row far longer than the rest (170000 scores: a cluster of 6 x 32768)
    dict(base="mtp_32k", batch=2, q_per_req=2, num_heads=16, topk=2048,
         seqlens=[170000, 3000], heavy="frac:0.01", seed=83),
    # another k, rows shorter than k next to a longer one
    dict(base="long_varlen", batch=3, q_per_req=1, num_heads=16, topk=100,
         seqlens=[5000, 90, 333], heavy="runs:0.005:8", seed=84),
    # many requests: most indexer CTAs score tiles of two of them
    dict(base="long_varlen", batch=40, q_per_req=1, num_heads=16, topk=2048,
         seqlens=(2000, 12000), heavy="runs:0.005:8", seed=86),
]


def _check_fused_selection(wl, g):
    T, k = wl.spec.num_tokens, wl.spec.topk
    sel = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    out = api.run_decode(g, topk_out=sel)
    logits = api.run_indexer(g)
    torch.cuda.synchronize()
    _assert_no_device_error()
    a = W.host_arrays(wl)
    vis = O.visible_lengths(a["seqlens"], a["q_per_req"])
    sel_np = sel.cpu().numpy()
    want = O.topk(logits.cpu().numpy(), vis, k)
    bad = [t for t in range(T) if not np.array_equal(sel_np[t], want[t])]
    assert not bad, f"rows {bad[:8]} differ from the top-k of the kernel's scores"
    o, _ = O.sparse_mla(a["q"], a["kv"], sel_np, a["page_table"], a["seqlens"], a["q_per_req"],
                        a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")
    return sel_np, logits


@pytest.mark.parametrize("case", SEL_CASES,
                         ids=["nq3", "nq4", "nq2-long-row", "k100", "b40"])
def test_fused_selection_matches_topk_of_the_scores(case):
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    if isinstance(seqlens, tuple):
        rng = np.random.default_rng(case["seed"])
        seqlens = rng.integers(seqlens[0], seqlens[1] + 1, size=case["batch"]).tolist()
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    _check_fused_selection(wl, g)


@pytest.mark.parametrize("nq", [1, 2])
def test_fused_selection_breaks_exact_ties_by_position(nq):
    """Index keys of zeros score exactly 0: with all but a few hundred keys
    zeroed, the k-th score is 0 and the selection must take the lowest
    positions among tens of thousands of equal scores (the top-k's tie
    resolution over positions, with candidate lists far beyond its shared
    memory); the last request's keys are all zero (every score ties)."""
    wl = W.make_workload(W.small_spec("long_varlen", batch=3, q_per_req=nq, num_heads=16,
                                      topk=2048, heavy="none", seed=85 + nq),
                         seqlens=[30000, 12000, 5000])
    rows = wl.k_fp8.shape[0]
    keep = torch.zeros(rows, dtype=torch.bool)
    keep[torch.from_numpy(np.random.default_rng(nq).choice(rows, 400, replace=False))] = True
    pt = wl.page_table[2]
    last = pt[pt >= 0].long()
    for pg in last.tolist():
        keep[pg * 64:(pg + 1) * 64] = False
    wl.layers[0].k_fp8[~keep] = 0
    g = wl.to("cuda")
    sel_np, logits = _check_fused_selection(wl, g)
    lg = logits.cpu().numpy()
    T = wl.spec.num_tokens
    vis = O.visible_lengths(wl.seqlens.numpy().astype(np.int64), nq)
    for t in range(T):
        kth = np.sort(lg[t, :vis[t]])[::-1][2047]
        assert kth == 0.0, "the threshold must lie among the zero scores"
    # the all-zero request selects its first k positions
    for t in range((T // 3) * 2, T):
        assert np.array_equal(sel_np[t], np.arange(2048))


# ---------------------------------------------------------------- cache write

def _new_tokens(T, seed):
    """New tokens' latent rows and indexer keys (bf16): mixed magnitudes, one
    key of zeros, one with values far above 448 before scaling."""
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn(T, 576, generator=g).to(torch.bfloat16)
    key = torch.randn(T, 128, generator=g) * torch.exp(torch.randn(T, 1, generator=g) * 2)
    key[0] = 0.0
    if T > 1:
        key[1] *= 1e4
    return lat, key.to(torch.bfloat16)


def _check_cache_write(wl, g, seed, whole_oracle):
    """Runs dsa_cache_write on the device copy g of wl and compares every
    byte of the written rows and a sample of the others with the oracle
    (its cache_write on the whole caches, or its per-row pieces when the
    caches are workload-sized)."""
    T, nq = wl.spec.num_tokens, wl.spec.q_per_req
    lat, key = _new_tokens(T, seed)
    lat_b, key_b = W.bf16_bits(lat), W.bf16_bits(key)
    table, seqlens = wl.page_table.numpy(), wl.seqlens.numpy()
    rows = [int(O.physical_rows(table[t // nq], [p])[0])
            for t, p in enumerate(O.new_token_positions(seqlens, nq))]
    rng = np.random.default_rng(seed)
    sample = np.unique(np.concatenate([rows, rng.integers(0, wl.kv.shape[0], 4096)]))
    if whole_oracle:
        want_kv, want_k8, want_ks = O.cache_write(lat_b, key_b, W.bf16_bits(wl.kv), wl.k_fp8.numpy(),
                                                  wl.k_scale.numpy(), table, seqlens, nq)
        want_kv, want_k8, want_ks = want_kv[sample], want_k8[sample], want_ks[sample]
    else:
        idx = torch.from_numpy(sample)
        want_kv = W.bf16_bits(wl.kv[idx]).copy()
        want_k8 = wl.k_fp8[idx].numpy().copy()
        want_ks = wl.k_scale[idx].numpy().copy()
        codes, scales = O.quantize_index_key(key_b)
        where = {int(r): n for n, r in enumerate(sample)}
        for t, r in enumerate(rows):
            want_kv[where[r]], want_k8[where[r]], want_ks[where[r]] = lat_b[t], codes[t], scales[t]
    api.dsa_cache_write(api.workload_desc(g), lat.cuda(), key.cuda(), g.kv, g.k_fp8, g.k_scale)
    _assert_no_device_error()
    didx = torch.from_numpy(sample).cuda()
    assert np.array_equal(W.bf16_bits(g.kv[didx]), want_kv)
    assert np.array_equal(g.k_fp8[didx].cpu().numpy(), want_k8)
    assert np.array_equal(g.k_scale[didx].cpu().numpy().view(np.uint32), want_ks.view(np.uint32))
    return rows


def test_cache_write_bit_exact_small():
    wl, g = _gpu_wl("mtp_32k", batch=5, q_per_req=3, num_heads=128, topk=64,
                    seqlens=[70, 129, 3, 640, 200], heavy="none", seed=81)
    rows = _check_cache_write(wl, g, 81, whole_oracle=True)
    assert len(set(rows)) == 15


@pytest.mark.parametrize("name", ["long_128k", "mtp_32k"])
def test_cache_write_bit_exact_workload_sized(name):
    wl = W.make_workload(name)
    g = wl.to("cuda")
    _check_cache_write(wl, g, 82, whole_oracle=False)


def test_cache_write_flags_bad_page_id():
    wl, g = _gpu_wl("long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[3000, 700], heavy="none", seed=83)
    g.page_table[1, (700 - 1) // 64] = -1                 # the new token's page
    lat, key = _new_tokens(2, 83)
    before = g.kv.clone()
    api.dsa_cache_write(api.workload_desc(g), lat.cuda(), key.cuda(), g.kv, g.k_fp8, g.k_scale)
    assert api.dsa_get_device_error() == 5               # DSA_ERR_DEVICE_CHECK
    row0 = int(O.physical_rows(wl.page_table.numpy()[0], [2999])[0])
    assert torch.equal(g.kv[row0], lat[0].cuda())         # the valid row is still written
    changed = (g.kv != before).any(dim=1).nonzero().flatten().tolist()
    assert changed == [row0]


FUSED_WRITE_CASES = [
    # 2049 with n_q = 2: the new tokens (2047, 2048) straddle the last two tiles
    dict(base="mtp_32k", batch=3, q_per_req=2, num_heads=128, topk=2048, seqlens=[5000, 2049, 9000],
         heavy="frac:0.01", seed=91),
    dict(base="long_varlen", batch=2, q_per_req=1, num_heads=128, topk=2048, seqlens=[20000, 12345],
         heavy="runs:0.005:8", seed=92),
    # 129 and 2048: requests whose queries select every token (no scan)
    dict(base="short_dense", batch=3, q_per_req=1, num_heads=128, topk=2048, seqlens=[129, 3000, 2048],
         heavy="none", seed=93),
]


@pytest.mark.parametrize("case", FUSED_WRITE_CASES, ids=lambda c: c["base"])
@pytest.mark.parametrize("given_selection", [False, True], ids=["indexer", "topk_in"])
def test_fused_layer_with_cache_write(case, given_selection):
    """dsa_decode_fused_write = the oracle's cache write, then the layer on
    the written caches.  Each new token's index key is ten times its own
    query's highest-weighted index head and its latent row four times a
    random one, so a stale key or row changes the selection or the output."""
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    T, k, nq = wl.spec.num_tokens, wl.spec.topk, wl.spec.q_per_req
    lat, _ = _new_tokens(T, case["seed"])
    lat = (lat.float() * 4).to(torch.bfloat16)
    qhat = wl.q_fp8.view(torch.float8_e4m3fn).float() * wl.q_scale[:, None, None]
    best = torch.argmax(wl.w, dim=1)
    key = (10 * qhat[torch.arange(T), best]).to(torch.bfloat16)
    a = W.host_arrays(wl)
    a["kv"], a["k_fp8"], a["k_scale"] = O.cache_write(
        W.bf16_bits(lat), W.bf16_bits(key), a["kv"], a["k_fp8"], a["k_scale"], a["page_table"],
        a["seqlens"], nq)
    vis = O.visible_lengths(a["seqlens"], nq)
    lc = g.layers[0]
    out = torch.empty((T, wl.spec.num_heads, 512), dtype=torch.float32, device="cuda")
    ws = api.alloc_workspace(g)
    if given_selection:
        sel_np = O.topk(np.random.default_rng(3).random((T, int(max(vis)))), vis, k)
        sel = torch.from_numpy(sel_np.astype(np.int32)).cuda()
        api.dsa_decode_fused_write(api.workload_desc(g), lat.cuda(), key.cuda(), g.q_fp8, g.q_scale,
                                   g.w, lc.k_fp8, lc.k_scale, lc.q, lc.kv, out, ws, g.max_seqlen,
                                   wl.spec.sm_scale, topk_in=sel)
    else:
        sel = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
        api.dsa_decode_fused_write(api.workload_desc(g), lat.cuda(), key.cuda(), g.q_fp8, g.q_scale,
                                   g.w, lc.k_fp8, lc.k_scale, lc.q, lc.kv, out, ws, g.max_seqlen,
                                   wl.spec.sm_scale, topk_out=sel)
    torch.cuda.synchronize()
    _assert_no_device_error()
    # the caches hold exactly the oracle's written rows
    rows = np.unique(np.concatenate([
        O.physical_rows(a["page_table"][t // nq], [p])
        for t, p in enumerate(O.new_token_positions(a["seqlens"], nq))]))
    ridx = torch.from_numpy(rows).cuda()
    assert np.array_equal(W.bf16_bits(lc.kv[ridx]), a["kv"][rows])
    assert np.array_equal(lc.k_fp8[ridx].cpu().numpy(), a["k_fp8"][rows])
    assert np.array_equal(lc.k_scale[ridx].cpu().numpy().view(np.uint32),
                          a["k_scale"][rows].view(np.uint32))
    if not given_selection:
        sel_np = sel.cpu().numpy()
        # the selection is the top-k of the written cache's scores
        I, E = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                                a["page_table"], a["seqlens"], nq)
        for t, n in enumerate(vis):
            chosen = sel_np[t][sel_np[t] >= 0]
            if n <= k:
                assert np.array_equal(chosen, np.arange(n))
                continue
            kth = np.sort(I[t, :n])[::-1][k - 1]
            assert (I[t, chosen] >= kth - 2 * IDX_REL * E[t, chosen]).all()
            assert n - 1 in chosen                      # the query's own new token
    o, _ = O.sparse_mla(a["q"], a["kv"], sel_np, a["page_table"], a["seqlens"], nq, a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")


def test_host_errors_are_returned_before_launch():
    wl, g = _gpu_wl("long_varlen", batch=1, q_per_req=1, num_heads=128, topk=2048,
                    seqlens=[300], heavy="none", seed=72)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.DSAError) as e:
        api.run_decode(g, ws=ws)
    assert e.value.status == 3                           # DSA_ERR_WORKSPACE
    d = api.workload_desc(g)
    d.num_heads = 100
    with pytest.raises(api.DSAError) as e:
        api.dsa_sparse_mla_decode_split(d, g.q, g.kv, torch.zeros((1, 2048), dtype=torch.int32, device="cuda"),
                                        1, 0.1, torch.empty((1, 100, 1, 512), device="cuda"),
                                        torch.empty((1, 100, 1), device="cuda"))
    assert e.value.status == 2                           # DSA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- workload sizes

def _sampled_checks(wl, g, sel, out, logits, rows_to_check, n_pos=4096):
    """Oracle checks on sampled outputs of a workload-sized run."""
    nq, k = wl.spec.q_per_req, wl.spec.topk
    seqlens = wl.seqlens.cpu().numpy()
    table = wl.page_table.cpu().numpy()
    vis = O.visible_lengths(seqlens, nq)
    sel_np = sel.cpu().numpy()
    lg = logits.cpu().numpy()
    # top-k: exact against the oracle on the kernel's scores, every row
    assert np.array_equal(sel_np, O.topk(lg, vis, k))
    rng = np.random.default_rng(0)
    for t in rows_to_check:
        r, n = t // nq, int(vis[t])
        pos = np.unique(np.concatenate([rng.integers(0, n, size=min(n_pos, n)),
                                        sel_np[t][sel_np[t] >= 0]]))
        rows = torch.from_numpy(O.physical_rows(table[r], pos)).cuda()
        k8 = wl.k_fp8[rows].cpu().numpy()
        ks = wl.k_scale[rows].cpu().numpy()
        I, E = O.indexer_logits_at(wl.q_fp8[t].cpu().numpy(), float(wl.q_scale[t]),
                                   wl.w[t].cpu().numpy(), k8, ks, np.arange(len(pos)))
        assert (np.abs(lg[t, pos] - I) <= IDX_REL * E).all()
        chosen = sel_np[t][sel_np[t] >= 0]
        lat = wl.kv[torch.from_numpy(O.physical_rows(table[r], chosen)).cuda()]
        o, _ = O.attend(W.bf16_bits(wl.q[t]), W.bf16_bits(lat), wl.spec.sm_scale)
        _assert_close_att(out[t].cpu().numpy(), o, f"row {t}")


def test_mli_layer_workload_sized():
    """dsa_decode_mli on the full mli_195k workload (4 requests of 196608
    tokens, two layers): layer 2's own selection equals the fused layer's on
    layer 2 bit for bit (rows of 196608 scores, selected beside the
    attention), and its output at sampled rows is the oracle's attention of
    layer 2's queries over layer 1's selection."""
    wl = W.make_workload("mli_195k", device="cuda")
    T, k, H = wl.spec.num_tokens, wl.spec.topk, wl.spec.num_heads
    desc = api.workload_desc(wl)
    sel1 = torch.empty((T, k), dtype=torch.int32, device="cuda")
    api.run_decode(wl, layer=0, topk_out=sel1)
    sel2_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
    api.run_decode(wl, layer=1, topk_out=sel2_ref)
    lc2 = wl.layers[1]
    sel2 = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    out = torch.full((T, H, 512), float("nan"), device="cuda")
    api.dsa_decode_mli(desc, wl.q_fp8, wl.q_scale, wl.w, lc2.k_fp8, lc2.k_scale, lc2.q, lc2.kv,
                       sel1, sel2, out, api.alloc_workspace(wl, 0), wl.max_seqlen,
                       wl.spec.sm_scale, 0)
    torch.cuda.synchronize()
    _assert_no_device_error()
    assert torch.equal(sel2, sel2_ref)
    table = wl.page_table.cpu().numpy()
    s1 = sel1.cpu().numpy()
    for t in sorted({0, T - 1}):
        chosen = s1[t][s1[t] >= 0]
        lat = lc2.kv[torch.from_numpy(O.physical_rows(table[t], chosen)).cuda()]
        o, _ = O.attend(W.bf16_bits(lc2.q[t]), W.bf16_bits(lat), wl.spec.sm_scale)
        _assert_close_att(out[t].cpu().numpy(), o, f"row {t}")
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["long_128k", "mtp_32k", "short_dense", "tiny_4k", "long_varlen",
                                  "mli_195k"])
def test_workload_sized_sampled(name):
    wl = W.make_workload(name, device="cuda")
    T, k = wl.spec.num_tokens, wl.spec.topk
    sel = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = api.run_decode(wl, topk_out=sel)
    logits = api.run_indexer(wl)
    _assert_no_device_error()
    check = sorted({0, T // 2, T - 1})
    _sampled_checks(wl, wl, sel, out, logits, check)
    del wl
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- FP8 latent cache

def _fp8_cache(g, layer=0):
    kv = g.layers[layer].kv
    kv8 = torch.empty((kv.shape[0], 656), dtype=torch.uint8, device="cuda")
    api.dsa_latent_to_fp8(kv, kv8)
    return kv8


def test_latent_to_fp8_bit_exact():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1000, 576)) * np.exp(rng.standard_normal((1000, 1)) * 3)
    x[0, :128] = 0.0                       # a tile of zeros: scale 1
    x[1, 128:256] *= 1e30                  # large magnitudes
    x[2, 300] *= -1e3                      # one outlier in a tile
    bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kv = torch.from_numpy(bits.view(np.int16)).cuda()
    kv8 = torch.empty((1000, 656), dtype=torch.uint8, device="cuda")
    api.dsa_latent_to_fp8(kv, kv8)
    torch.cuda.synchronize()
    assert np.array_equal(kv8.cpu().numpy(), O.quantize_latent(bits))


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("case", MLA_CASES, ids=lambda c: f"{c['base']}-H{c['num_heads']}-k{c['topk']}")
def test_sparse_mla_fp8_split_and_merge_match_oracle(case, splits):
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, heavy="none", **case)
    a, idx = _oracle_indices(wl)
    kv8 = _fp8_cache(g)
    kv8_h = kv8.cpu().numpy()
    assert np.array_equal(kv8_h, O.quantize_latent(a["kv"]))
    desc = api.workload_desc(g)
    S = api.dsa_num_splits_auto(desc) if splits == 0 else splits
    T, H = wl.spec.num_tokens, wl.spec.num_heads
    mid_o = torch.empty((T, H, S, 512), dtype=torch.float32, device="cuda")
    mid_lse = torch.empty((T, H, S), dtype=torch.float32, device="cuda")
    api.dsa_sparse_mla_decode_split_fp8(desc, g.layers[0].q, kv8,
                                        torch.from_numpy(idx.astype(np.int32)).cuda(), S,
                                        wl.spec.sm_scale, mid_o, mid_lse)
    out, lse = api.run_merge(mid_o, mid_lse)
    _assert_no_device_error()
    mo, ml = O.sparse_mla_split(a["q"], None, idx, a["page_table"], a["seqlens"], a["q_per_req"],
                                a["sm_scale"], S, kv_fp8=kv8_h)
    _assert_close_att(mid_o.cpu().numpy(), mo, "Mid_O")
    _assert_close_att(mid_lse.cpu().numpy(), ml, "Mid_LSE")
    o, l = O.sparse_mla_fp8(a["q"], kv8_h, idx, a["page_table"], a["seqlens"], a["q_per_req"],
                            a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")
    _assert_close_att(lse.cpu().numpy(), l, "LSE")


@pytest.mark.parametrize("case", FUSED_CASES, ids=lambda c: c["base"])
def test_fused_layer_fp8_latent(case):
    """The layer over the FP8 latent cache: the same selection as the bf16
    layer (the indexer and top-k do not read the latent cache), and the
    attention over the dequantised rows."""
    case = dict(case)
    base, seqlens = case.pop("base"), case.pop("seqlens")
    wl, g = _gpu_wl(base, seqlens=seqlens, **case)
    T, k, H = wl.spec.num_tokens, wl.spec.topk, wl.spec.num_heads
    kv8 = _fp8_cache(g)
    sel16 = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    api.run_decode(g, topk_out=sel16)
    sel8 = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.float32, device="cuda")
    lc = g.layers[0]
    api.dsa_decode_fused_fp8kv(api.workload_desc(g), g.q_fp8, g.q_scale, g.w, lc.k_fp8, lc.k_scale,
                               lc.q, kv8, out, api.alloc_workspace(g), g.max_seqlen,
                               wl.spec.sm_scale, topk_out=sel8)
    torch.cuda.synchronize()
    _assert_no_device_error()
    assert torch.equal(sel8, sel16)
    a = W.host_arrays(wl)
    o, _ = O.sparse_mla_fp8(a["q"], kv8.cpu().numpy(), sel8.cpu().numpy(), a["page_table"],
                            a["seqlens"], a["q_per_req"], a["sm_scale"])
    _assert_close_att(out.cpu().numpy(), o, "O")


@pytest.mark.parametrize("name", ["long_128k", "mtp_32k", "short_dense"])
def test_fused_layer_fp8_latent_workload_sized(name):
    wl = W.make_workload(name, device="cuda")
    T, k, H = wl.spec.num_tokens, wl.spec.topk, wl.spec.num_heads
    kv8 = _fp8_cache(wl)
    sel = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, 512), dtype=torch.float32, device="cuda")
    lc = wl.layers[0]
    api.dsa_decode_fused_fp8kv(api.workload_desc(wl), wl.q_fp8, wl.q_scale, wl.w, lc.k_fp8,
                               lc.k_scale, lc.q, kv8, out, api.alloc_workspace(wl), wl.max_seqlen,
                               wl.spec.sm_scale, topk_out=sel)
    torch.cuda.synchronize()
    _assert_no_device_error()
    table = wl.page_table.cpu().numpy()
    sel_np = sel.cpu().numpy()
    for t in sorted({0, T // 2, T - 1}):
        r = t // wl.spec.q_per_req
        chosen = sel_np[t][sel_np[t] >= 0]
        rows = torch.from_numpy(O.physical_rows(table[r], chosen)).cuda()
        # spot-check the stored rows against the oracle's quantisation
        assert np.array_equal(kv8[rows[:64]].cpu().numpy(),
                              O.quantize_latent(W.bf16_bits(lc.kv[rows[:64]])))
        o, _ = O.attend_fp8(W.bf16_bits(lc.q[t]), kv8[rows].cpu().numpy(), wl.spec.sm_scale)
        _assert_close_att(out[t].cpu().numpy(), o, f"row {t}")
    del wl
    torch.cuda.empty_cache()
