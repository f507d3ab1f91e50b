"""Pins of the float64 oracle to things other than itself (CPU only).

Each test checks the oracle against printed values on the pages, a library
routine for a special case, a brute-force computation on tiny inputs, an
invariance or a closed form, chosen so that a plausible slip in the oracle (a
dropped ReLU, a wrong scale, a transposed page index, a reversed tie rule, a
wrong visibility offset, a dropped softmax term) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from deepseek_sparse_attention_lightning_gb300 import workloads as W


def _read_golden(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- formats

def test_e4m3_decode_matches_torch_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(b)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2                       # 0x7F and 0xFF only
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_bf16_decode_matches_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.decode_bf16(bits), x.to(torch.float64).numpy())


def test_e4m3_encode_matches_torch_in_range():
    # random magnitudes over the whole finite range, every code's value, and
    # every midpoint between neighbouring codes (ties go to the even mantissa)
    rng = np.random.default_rng(3)
    vals = O.decode_e4m3(np.arange(0x7F, dtype=np.uint8))          # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 20000))
    x = np.concatenate([vals, mids, rand, rand * 0.999, 2.0 ** -10 * rng.random(1000)])
    x = np.concatenate([x, -x]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.encode_e4m3(x), ref)


def test_e4m3_encode_saturates_and_keeps_sign():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e30, -1e30, -0.0, 0.0])
    assert O.encode_e4m3(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00]


def test_index_key_quantisation_bound_and_amax():
    rng = np.random.default_rng(4)
    k = torch.from_numpy(rng.standard_normal((64, 128)) * rng.uniform(0.01, 30, (64, 1)))
    kb = k.to(torch.bfloat16)
    bits = kb.view(torch.int16).numpy().view(np.uint16)
    codes, scale = O.quantize_index_key(bits)
    kf = kb.to(torch.float64).numpy()
    assert np.allclose(scale, np.abs(kf).max(axis=1) / 448.0, rtol=1e-7, atol=0)
    x = kf / scale[:, None]
    err = np.abs(O.decode_e4m3(codes) - x)
    # round to nearest: half a step of 3 mantissa bits, or of the subnormal grid
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))
    # the largest magnitude of each token lands on +-448
    am = np.abs(kf).argmax(axis=1)
    assert set(codes[np.arange(64), am].tolist()) <= {0x7E, 0xFE}
    # a token of zeros: zero codes, scale 1
    c0, s0 = O.quantize_index_key(np.zeros((1, 128), np.uint16))
    assert not c0.any() and s0[0] == 1.0


# ---------------------------------------------------------------- geometry

def test_visible_lengths_worked_example(golden_dir):
    g = {r[0]: r[1:] for r in _read_golden(golden_dir, "mtp_visible_lengths.txt")}
    nq, s = int(g["q_per_req"][0]), int(g["seqlen"][0])
    want = [int(v) for v in g["visible"]]
    assert O.visible_lengths([s], nq).tolist() == want
    # two requests keep request-major order
    assert O.visible_lengths([s, 5], nq).tolist() == want + [3, 4, 5]


def test_physical_rows_follow_page_table():
    table = np.array([7, 2, 9])
    pos = np.array([0, 63, 64, 130])
    assert O.physical_rows(table, pos).tolist() == [7 * 64, 7 * 64 + 63, 2 * 64, 9 * 64 + 2]


def test_new_token_positions_are_the_last_visible(golden_dir):
    # the new tokens are the last q_per_req of the request: token i sits at
    # the position just before what query i sees (worked example: 7, 8, 9)
    g = {r[0]: r[1:] for r in _read_golden(golden_dir, "mtp_visible_lengths.txt")}
    nq, s = int(g["q_per_req"][0]), int(g["seqlen"][0])
    want = [int(v) - 1 for v in g["visible"]]
    assert O.new_token_positions([s], nq).tolist() == want
    assert O.new_token_positions([s, 5], nq).tolist() == want + [2, 3, 4]


def test_cache_write_touches_only_the_new_rows():
    rng = np.random.default_rng(6)
    B, nq, pages = 3, 2, 12
    table = rng.permutation(pages).reshape(B, 4).astype(np.int32)
    seqlens = np.array([70, 129, 2])
    kv = rng.integers(0, 65535, (pages * 64, 576), dtype=np.uint16)
    kf8 = rng.integers(0, 255, (pages * 64, 128), dtype=np.uint8)
    ksc = rng.random(pages * 64).astype(np.float32)
    lat = rng.integers(0, 65535, (B * nq, 576), dtype=np.uint16)
    key = torch.randn(B * nq, 128, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    kbits = key.view(torch.int16).numpy().view(np.uint16)
    kv2, kf2, ks2 = O.cache_write(lat, kbits, kv, kf8, ksc, table, seqlens, nq)
    rows = []
    for t, p in enumerate(O.new_token_positions(seqlens, nq)):
        r = t // nq
        row = table[r][p // 64] * 64 + p % 64
        rows.append(row)
        assert np.array_equal(kv2[row], lat[t])
        deq = O.decode_e4m3(kf2[row]) * ks2[row]
        assert np.allclose(deq, key[t].to(torch.float64).numpy(), rtol=0.07, atol=ks2[row] * 2.0 ** -9)
    other = np.setdiff1d(np.arange(pages * 64), rows)
    assert np.array_equal(kv2[other], kv[other]) and np.array_equal(kf2[other], kf8[other])
    assert np.array_equal(ks2[other], ksc[other])
    assert len(set(rows)) == B * nq


# ---------------------------------------------------------------- indexer

def _small(**kw):
    base = dict(batch=2, q_per_req=2, num_heads=16, topk=64, seqlen=(200, 330),
                heavy="count:8", paged=True, seed=11)
    base.update(kw)
    return W.make_workload(W.small_spec("mtp_32k", **base))


def _logits(a, **over):
    d = dict(a)
    d.update(over)
    return O.indexer_logits(d["q_fp8"], d["q_scale"], d["w"], d["k_fp8"], d["k_scale"],
                            d["page_table"], d["seqlens"], d["q_per_req"])


def test_indexer_head_permutation_invariance():
    a = W.host_arrays(_small())
    I, _ = _logits(a)
    perm = np.random.default_rng(0).permutation(O.INDEX_HEADS)
    I2, _ = _logits(a, q_fp8=a["q_fp8"][:, perm], w=a["w"][:, perm])
    fin = np.isfinite(I)
    assert np.allclose(I[fin], I2[fin], rtol=1e-12, atol=1e-12)
    # a permutation of the weights alone changes the scores
    I3, _ = _logits(a, w=a["w"][:, perm])
    assert not np.allclose(I[fin], I3[fin])


def test_indexer_page_table_equivariance():
    wl = _small(paged=False)
    a = W.host_arrays(wl)
    I, _ = _logits(a)
    # move every physical page elsewhere and rewrite the table to match
    npg = wl.num_pages
    perm = np.random.default_rng(1).permutation(npg)        # old page p -> new page perm[p]
    k8 = np.empty_like(a["k_fp8"])
    ks = np.empty_like(a["k_scale"])
    for p in range(npg):
        k8[perm[p] * 64:(perm[p] + 1) * 64] = a["k_fp8"][p * 64:(p + 1) * 64]
        ks[perm[p] * 64:(perm[p] + 1) * 64] = a["k_scale"][p * 64:(p + 1) * 64]
    table = np.where(a["page_table"] >= 0, perm[np.maximum(a["page_table"], 0)], -1)
    I2, _ = _logits(a, k_fp8=k8, k_scale=ks, page_table=table)
    assert np.array_equal(I, I2)


def test_indexer_scale_homogeneity():
    a = W.host_arrays(_small())
    I, _ = _logits(a)
    I_k, _ = _logits(a, k_scale=a["k_scale"] * 2.0)
    I_q, _ = _logits(a, q_scale=a["q_scale"] * 4.0)
    fin = np.isfinite(I)
    assert np.allclose(I_k[fin], 2.0 * I[fin], rtol=1e-13, atol=0)
    assert np.allclose(I_q[fin], 4.0 * I[fin], rtol=1e-13, atol=0)


def test_indexer_relu_makes_nonnegative_weights_give_nonnegative_scores():
    a = W.host_arrays(_small())
    wpos = np.abs(a["w"])
    I, _ = _logits(a, w=wpos)
    fin = np.isfinite(I)
    assert (I[fin] >= 0).all()
    # and the data do contain negative head dots, so the ReLU mattered:
    qhat = O.decode_e4m3(a["q_fp8"][0]) * a["q_scale"][0]
    khat = O.decode_e4m3(a["k_fp8"][:64]) * a["k_scale"][:64, None]
    assert (khat @ qhat.T < 0).mean() > 0.3
    I_neg, _ = _logits(a, w=-wpos)
    assert (I_neg[fin] <= 0).all()


def test_indexer_sum_of_relus_closed_form():
    # head 0 query = the key, head 1 query = minus the key, w = (1, 1, 0, ...):
    # sum_j w_j ReLU(q_j . k) = ReLU(|k|^2) + ReLU(-|k|^2) = |k|^2 (scaled);
    # ReLU of the weighted sum would give 0 instead.
    rng = np.random.default_rng(3)
    k8 = rng.integers(0, 0x7E, size=(64, 128), dtype=np.uint8)  # finite bytes
    q8 = np.zeros((1, 64, 128), dtype=np.uint8)
    q8[0, 0] = k8[5]
    q8[0, 1] = k8[5] ^ 0x80                                     # flip the sign bit
    w = np.zeros((1, 64))
    w[0, 0] = w[0, 1] = 1.0
    sq, sk = np.array([0.5]), np.full(64, 0.25)
    I, E = O.indexer_logits(q8, sq, w, k8, sk, np.array([[0]]), np.array([64]), 1)
    kv = O.decode_e4m3(k8[5])
    assert I[0, 5] == pytest.approx(float(kv @ kv) * 0.5 * 0.25, rel=1e-14)
    assert E[0, 5] == pytest.approx(2 * float(kv @ kv) * 0.5 * 0.25, rel=1e-14)


def test_indexer_positive_case_is_a_matrix_vector_product():
    # with every FP8 value positive all head dots are positive, the ReLU is the
    # identity and I = khat . (sum_j w_j qhat_j): one library matvec.
    rng = np.random.default_rng(4)
    k8 = rng.integers(0x08, 0x70, size=(128, 128), dtype=np.uint8)
    q8 = rng.integers(0x08, 0x70, size=(1, 64, 128), dtype=np.uint8)
    w = rng.random((1, 64))
    sq, sk = np.array([0.01]), rng.random(128) + 0.5
    I, E = O.indexer_logits(q8, sq, w, k8, sk, np.array([[0, 1]]), np.array([128]), 1)
    khat = O.decode_e4m3(k8) * sk[:, None]
    qsum = np.einsum("j,jd->d", w[0], O.decode_e4m3(q8[0]) * sq[0])
    ref = np.dot(khat, qsum)
    assert np.allclose(I[0], ref, rtol=1e-12)
    assert np.allclose(E[0], I[0], rtol=1e-12)     # all terms positive: bound == value


def test_indexer_masks_invisible_positions_and_bound_dominates():
    wl = _small()
    a = W.host_arrays(wl)
    I, E = _logits(a)
    vis = O.visible_lengths(a["seqlens"], a["q_per_req"])
    for t, n in enumerate(vis):
        assert np.isfinite(I[t, :n]).all()
        assert np.isneginf(I[t, n:]).all()
    fin = np.isfinite(I)
    assert (E[fin] >= np.abs(I[fin]) * (1 - 1e-12)).all()


def test_planted_heavy_tokens_score_high():
    wl = W.make_workload(W.small_spec("tiny_4k", seqlen=1024, topk=128, heavy="count:16"))
    a = W.host_arrays(wl)
    I, _ = _logits(a)
    heavy = wl.heavy[0]
    rank = (I[0][None, :] > I[0][heavy][:, None]).sum(axis=1)
    assert (rank < 0.01 * 1024 + len(heavy)).all()


# ---------------------------------------------------------------- top-k

def _brute_topk(row, n, k):
    order = sorted(range(n), key=lambda i: (-float(row[i]), i))
    return sorted(order[:min(k, n)])


@pytest.mark.parametrize("n", [1, 5, 17, 64])
def test_topk_matches_brute_force_sort(n):
    rng = np.random.default_rng(n)
    for k in {1, 3, max(1, n - 1), n, n + 5}:
        # few distinct values so that ties are frequent
        scores = rng.integers(-4, 5, size=(3, 80)).astype(np.float32) * 0.5
        vis = np.array([n, max(0, n - 2), n])
        got = O.topk(scores, vis, k)
        for t in range(3):
            want = _brute_topk(scores[t], int(vis[t]), k)
            m = len(want)
            assert got[t, :m].tolist() == want
            assert (got[t, m:] == -1).all()


def test_topk_ties_go_to_lower_index_and_signed_zero_is_equal():
    scores = np.zeros((2, 10), dtype=np.float32)
    scores[1, ::2] = -0.0
    got = O.topk(scores, np.array([10, 10]), 4)
    assert got[0].tolist() == [0, 1, 2, 3]
    assert got[1].tolist() == [0, 1, 2, 3]


def test_topk_selects_everything_when_k_exceeds_visible():
    scores = np.random.default_rng(2).standard_normal((2, 50)).astype(np.float32)
    got = O.topk(scores, np.array([50, 20]), 64)
    assert got[0, :50].tolist() == list(range(50)) and (got[0, 50:] == -1).all()
    assert got[1, :20].tolist() == list(range(20)) and (got[1, 20:] == -1).all()


# ---------------------------------------------------------------- sparse MLA

def _mla_inputs(seqlens=(90, 130), nq=1, H=16, seed=7):
    wl = W.make_workload(W.small_spec("mtp_32k", batch=len(seqlens), q_per_req=nq,
                                      num_heads=H, topk=256, heavy="none", seed=seed),
                         seqlens=list(seqlens))
    return wl, W.host_arrays(wl)


def test_sparse_mla_all_selected_equals_dense_sdpa():
    wl, a = _mla_inputs(seqlens=(90, 130), nq=2)
    vis = O.visible_lengths(a["seqlens"], 2)
    k = 256                                             # k >= every visible length
    idx = np.full((len(vis), k), -1)
    for t, n in enumerate(vis):
        idx[t, :n] = np.arange(n)
    out, lse = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 2, a["sm_scale"])
    for t, n in enumerate(vis):
        r = t // 2
        rows = O.physical_rows(a["page_table"][r], np.arange(n))
        lat = torch.from_numpy(O.decode_bf16(a["kv"][rows]))          # [n, 576]
        q = torch.from_numpy(O.decode_bf16(a["q"][t]))                 # [H, 576]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], lat[None, None].expand(1, q.shape[0], n, 576),
            lat[None, None, :, :512].expand(1, q.shape[0], n, 512), scale=a["sm_scale"])
        assert np.allclose(out[t], ref[0, :, 0].numpy(), rtol=1e-10, atol=1e-12)
        ref_lse = torch.logsumexp(a["sm_scale"] * (q @ lat.T), dim=1).numpy()
        assert np.allclose(lse[t], ref_lse, rtol=1e-12)


def test_decode_layer_with_k_covering_the_context_is_dense_attention():
    # The whole layer (indexer -> top-k -> sparse MLA) with k >= every visible
    # length selects every visible token, so its output is dense softmax
    # attention over the request, as torch computes it.
    wl, a = _mla_inputs(seqlens=(70, 129), nq=2, seed=11)
    res = O.decode_layer(a)
    vis = O.visible_lengths(a["seqlens"], 2)
    for t, n in enumerate(vis):
        assert np.array_equal(res["idx"][t][:n], np.arange(n)) and (res["idx"][t][n:] == -1).all()
        rows = O.physical_rows(a["page_table"][t // 2], np.arange(n))
        lat = torch.from_numpy(O.decode_bf16(a["kv"][rows]))
        q = torch.from_numpy(O.decode_bf16(a["q"][t]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, None, :], lat[None, None].expand(1, q.shape[0], n, 576),
            lat[None, None, :, :512].expand(1, q.shape[0], n, 512), scale=a["sm_scale"])
        assert np.allclose(res["out"][t], ref[0, :, 0].numpy(), rtol=1e-10, atol=1e-12)


def test_decode_layer_selects_the_best_fp32_scores():
    # With k below the visible length: k tokens per row, each with an fp32
    # score at least that of every visible token left out.
    wl, a = _mla_inputs(seqlens=(300, 517), nq=1, seed=12)
    a = dict(a, topk=64)
    res = O.decode_layer(a)
    vis = O.visible_lengths(a["seqlens"], 1)
    for t, n in enumerate(vis):
        sel = res["idx"][t][res["idx"][t] >= 0]
        assert len(sel) == 64 and len(np.unique(sel)) == 64 and (sel < n).all()
        sc = res["scores"][t, :n].astype(np.float32)
        out = np.setdiff1d(np.arange(n), sel)
        assert sc[sel].min() >= sc[out].max()


def test_sparse_mla_index_order_invariance_and_padding():
    wl, a = _mla_inputs(seqlens=(300,), nq=1)
    rng = np.random.default_rng(9)
    sel = np.sort(rng.choice(300, size=40, replace=False))
    idx = np.full((1, 64), -1)
    idx[0, :40] = sel
    o1, l1 = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    idx2 = idx.copy()
    idx2[0, :40] = rng.permutation(sel)
    o2, l2 = O.sparse_mla(a["q"], a["kv"], idx2, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14) and np.allclose(l1, l2, rtol=1e-13)
    # a different set gives a different result (the test can fail)
    idx3 = idx.copy()
    idx3[0, 0] = [i for i in range(300) if i not in set(sel)][0]
    o3, _ = O.sparse_mla(a["q"], a["kv"], idx3, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    assert not np.allclose(o1, o3)


def test_sparse_mla_single_token_closed_form():
    wl, a = _mla_inputs(seqlens=(100,), nq=1)
    idx = np.full((1, 64), -1)
    idx[0, 0] = 37
    out, lse = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 1, a["sm_scale"])
    row = O.decode_bf16(a["kv"][O.physical_rows(a["page_table"][0], [37])[0]])
    q = O.decode_bf16(a["q"][0])
    assert np.allclose(out[0], np.broadcast_to(row[:512], out[0].shape), rtol=0, atol=1e-15)
    assert np.allclose(lse[0], a["sm_scale"] * (q @ row), rtol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 7, 32])
def test_split_then_merge_equals_single_pass(splits):
    wl, a = _mla_inputs(seqlens=(700, 1500), nq=2, seed=13)
    vis = O.visible_lengths(a["seqlens"], 2)
    k = 2048
    rng = np.random.default_rng(splits)
    idx = np.full((len(vis), k), -1)
    for t, n in enumerate(vis):
        m = min(k, n, 1200)                      # some rows shorter than k
        idx[t, :m] = rng.choice(n, size=m, replace=False)
    o, l = O.sparse_mla(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 2, a["sm_scale"])
    mo, ml = O.sparse_mla_split(a["q"], a["kv"], idx, a["page_table"], a["seqlens"], 2,
                                a["sm_scale"], splits)
    om, lm = O.merge(mo, ml)
    assert np.allclose(om, o, rtol=1e-12, atol=1e-12)
    assert np.allclose(lm, l, rtol=1e-12, atol=1e-12)


def test_split_bounds_cover_positions_once():
    for k, s, n in [(2048, 9, 2048), (2048, 32, 1000), (100, 7, 100), (2048, 1, 5)]:
        b = O.split_bounds(k, s, n)
        covered = np.concatenate([np.arange(lo, hi) for lo, hi in b])
        assert covered.tolist() == list(range(n))
        assert all((lo % 64 == 0) or lo == n for lo, _ in b)


def test_merge_ignores_empty_splits():
    rng = np.random.default_rng(0)
    mo = rng.standard_normal((3, 2, 512))
    ml = np.array([[0.3, -np.inf], [-np.inf, -np.inf], [-np.inf, 1.5]])
    o, l = O.merge(mo, ml)
    assert np.allclose(o[0], mo[0, 0]) and l[0] == pytest.approx(0.3)
    assert np.allclose(o[1], 0.0) and np.isneginf(l[1])
    assert np.allclose(o[2], mo[2, 1]) and l[2] == pytest.approx(1.5)


# ---------------------------------------------------------------- cost model

def test_cost_model_reproduces_printed_table(golden_dir):
    rows = _read_golden(golden_dir, "cost_model_table.txt")
    table = [r for r in rows if r[0].isdigit()]
    named = {r[0]: float(r[1]) for r in rows if not r[0].isdigit()}
    assert len(table) == 3
    for L, dg, sg, cr, dm, sm, rr in table:
        L = int(L)
        dense_f, dsa_f = O.dense_decode_flops(L), O.decode_flops(L)
        dense_b, dsa_b = O.dense_decode_bytes(L), O.decode_bytes(L)
        assert f"{dense_f / 1e9:.2f}" == dg and f"{dsa_f / 1e9:.2f}" == sg
        assert f"{dense_f / dsa_f:.1f}" == cr
        assert f"{dense_b / 2 ** 20:.1f}" == dm and f"{dsa_b / 2 ** 20:.1f}" == sm
        assert f"{dense_b / dsa_b:.1f}" == rr
    assert round(O.pair_flops_mla() / 1e3) == named["pair_mla_kflops"]
    assert round(O.pair_flops_indexer() / 1e3) == named["pair_indexer_kflops"]
    assert round(100 * O.token_bytes_index() / O.token_bytes_latent()) == named["index_cache_overhead_pct"]


def test_layer_bytes_single_query_matches_cost_model():
    for L in (4096, 32768, 131072):
        assert O.layer_bytes([L], 1, 2048) == O.decode_bytes(L)
        fi, fa = O.layer_flops([L], 1, 2048, 128)
        assert fi + fa == O.decode_flops(L)


# ---------------------------------------------------------------- FP8 latent cache

def _bf16_bits(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_latent_fp8_layout_and_error_bound():
    # 656-byte rows: codes of dims 0..511, four fp32 scales, the rope bits.
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 576)) * np.exp(rng.standard_normal((9, 1)) * 3)
    x[0, :128] = 0.0                                    # a tile of zeros
    bits = _bf16_bits(x)
    q8 = O.quantize_latent(bits)
    assert q8.shape == (9, 656) and q8.dtype == np.uint8
    xv = O.decode_bf16(bits)
    # rope: the bf16 bit patterns, little-endian, bit for bit
    assert np.array_equal(q8[:, 528:].copy().view("<u2"), bits[:, 512:])
    sc = q8[:, 512:528].copy().view("<f4").astype(np.float64)
    tiles = xv[:, :512].reshape(9, 4, 128)
    amax = np.abs(tiles).max(axis=2)
    assert sc[0, 0] == 1.0                              # zeros: scale 1
    np.testing.assert_allclose(sc[amax > 0], amax[amax > 0] / 448.0, rtol=1e-6)
    # each tile's largest magnitude is code +-448 (0x7E / 0xFE)
    for n in range(1, 9):
        for g in range(4):
            j = int(np.argmax(np.abs(tiles[n, g])))
            assert q8[n, 128 * g + j] & 0x7F == 0x7E
            assert (q8[n, 128 * g + j] >> 7) == (tiles[n, g, j] < 0)
    # dequantised values: within half an E4M3 step of the input (relative
    # 2^-4 for normal codes, 2^-10 x scale for subnormal ones)
    d = O.dequantize_latent(q8)
    assert np.array_equal(d[:, 512:], xv[:, 512:])
    err = np.abs(d[:, :512] - xv[:, :512]).reshape(9, 4, 128)
    bound = np.maximum(np.abs(tiles) * 2.0 ** -4, sc[:, :, None] * 2.0 ** -10) * (1 + 1e-9)
    assert (err <= bound).all()
    # a dims shift or transposed tile would break these: dim 200 of row 3
    assert abs(d[3, 200] - xv[3, 200]) <= max(abs(xv[3, 200]) * 2 ** -4, sc[3, 1] * 2 ** -10)


def test_latent_fp8_attention_equals_bf16_when_exact():
    # Tiles made of E4M3 values times a power of two, each holding +-448 x 2^e:
    # the scale is 2^e exactly, quantisation is lossless, and the attention
    # over the FP8 cache equals the attention over the bf16 cache.
    rng = np.random.default_rng(6)
    rows = 64 * 3
    e4 = O.e4m3_table()[:0x7F]
    codes = rng.integers(0, 0x7F, size=(rows, 4, 128))
    signs = rng.choice([-1.0, 1.0], size=(rows, 4, 128))
    vals = e4[codes] * signs
    vals[:, :, 0] = 448.0 * rng.choice([-1.0, 1.0], size=(rows, 4))
    expo = rng.integers(-12, -6, size=(rows, 4, 1)).astype(np.float64)
    lat = np.concatenate([(vals * 2.0 ** expo).reshape(rows, 512),
                          rng.standard_normal((rows, 64))], axis=1)
    kv = _bf16_bits(lat)
    q8 = O.quantize_latent(kv)
    assert np.array_equal(O.dequantize_latent(q8), O.decode_bf16(kv))
    T, H = 2, 8
    q = _bf16_bits(rng.standard_normal((T, H, 576)) * 40)
    table = np.array([[2, 0, 1], [1, 2, 0]], dtype=np.int64)
    seqlens = np.array([150, 192])
    idx = np.full((T, 64), -1, dtype=np.int64)
    idx[0, :40] = rng.choice(150, 40, replace=False)
    idx[1, :64] = rng.choice(192, 64, replace=False)
    o1, l1 = O.sparse_mla(q, kv, idx, table, seqlens, 1, 0.07)
    o2, l2 = O.sparse_mla_fp8(q, q8, idx, table, seqlens, 1, 0.07)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)
    # and the FP8 split partials merge to the same output
    mo, ml = O.sparse_mla_split(q, None, idx, table, seqlens, 1, 0.07, 3, kv_fp8=q8)
    om, lm = O.merge(mo, ml)
    np.testing.assert_allclose(om, o1, rtol=0, atol=1e-10)
