"""Host-side checks of the C ABI (no GPU needed: no call here reaches a kernel).

The library is built with nvcc (it cross-compiles sm_103a without a GPU);
these tests check that it loads, exports every function include/dsa.h declares,
and rejects bad arguments on the host before anything is launched.
"""
import ctypes
import os
import re

import pytest
import torch

from deepseek_sparse_attention_lightning_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def _fake_desc(**over):
    d = dict(batch=2, q_per_req=1, num_heads=128, topk=2048, page_size=64, max_pages=4,
             num_pages=8, seqlens=0x10000, page_table=0x20000)
    d.update(over)
    return api.DecodeDesc(**d)


FAKE = 0x7f0000000000      # a 256-byte aligned, never dereferenced "device" pointer


def test_header_declares_the_hot_path_calls():
    names = _declared_functions()
    for n in ["dsa_indexer_logits", "dsa_topk", "dsa_sparse_mla_decode_split", "dsa_merge",
              "dsa_decode_fused", "dsa_workspace_bytes", "dsa_get_device_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_version(L):
    assert api.dsa_status_str(0) == "DSA_OK"
    assert api.dsa_status_str(5) == "DSA_ERR_DEVICE_CHECK"
    assert api.dsa_status_str(6) == "DSA_ERR_TIMEOUT"
    assert "sm_103a" in api.dsa_version()


def test_descriptor_validation(L):
    call = lambda d: L.dsa_indexer_logits(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, None)
    assert L.dsa_indexer_logits(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, None) == 1
    assert call(ctypes.byref(_fake_desc(batch=0))) == 1
    assert call(ctypes.byref(_fake_desc(seqlens=None))) == 1
    assert call(ctypes.byref(_fake_desc(page_table=0x20002))) == 1          # misaligned
    assert call(ctypes.byref(_fake_desc(num_heads=100))) == 2
    assert call(ctypes.byref(_fake_desc(num_heads=256))) == 2
    assert call(ctypes.byref(_fake_desc(page_size=32))) == 2
    assert call(ctypes.byref(_fake_desc(topk=4096))) == 2
    assert call(ctypes.byref(_fake_desc(q_per_req=5))) == 2
    assert call(ctypes.byref(_fake_desc(batch=2000))) == 2
    # logits leading dimension shorter than the page table covers
    assert L.dsa_indexer_logits(ctypes.byref(_fake_desc()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                128, None) == 1
    assert L.dsa_indexer_logits(ctypes.byref(_fake_desc()), FAKE + 1, FAKE, FAKE, FAKE, FAKE, FAKE,
                                256, None) == 1


def test_workspace_checks(L):
    d = ctypes.byref(_fake_desc())
    assert L.dsa_topk(d, FAKE, 256, FAKE, FAKE, 16, None) == 3
    assert L.dsa_topk(d, FAKE, 256, FAKE, None, 1 << 30, None) == 3
    need = L.dsa_topk_workspace_bytes(d, 256)
    assert need > 0
    n1 = L.dsa_workspace_bytes(d, 256, 1)
    n2 = L.dsa_workspace_bytes(d, 256, 4)
    assert 0 < n1 < n2
    assert L.dsa_workspace_bytes(d, 0, 1) == 0
    assert L.dsa_decode_fused(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0.07, 1, 256,
                              FAKE, FAKE, n1 - 1, None) == 3
    # max_seqlen beyond what the page table can hold
    assert L.dsa_decode_fused(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0.07, 1, 257,
                              FAKE, FAKE, n1, None) == 1
    # bad scale / split count
    assert L.dsa_decode_fused(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, -1.0, 1, 256,
                              FAKE, FAKE, n1, None) == 1
    assert L.dsa_sparse_mla_decode_split(d, FAKE, FAKE, FAKE, 33, 0.07, FAKE, FAKE, None) == 1
    # the layer with the cache write: a misaligned new latent row, a short workspace
    assert L.dsa_decode_fused_write(d, FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    None, None, 0.07, 1, 256, FAKE, FAKE, n1, None) == 1
    assert L.dsa_decode_fused_write(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                    None, None, 0.07, 1, 256, FAKE, FAKE, n1 - 1, None) == 3


def test_step_layout(L):
    B, nq, H, mp = 3, 2, 128, 5
    lay = api.dsa_step_layout_get(B, nq, H, mp)
    T = B * nq
    need = [("q_fp8", T * 64 * 128), ("q_scale", T * 4), ("w", T * 64 * 4),
            ("q", T * H * 576 * 2), ("seqlens", B * 4), ("page_table", B * mp * 4)]
    end = 0
    for name, nbytes in need:
        off = getattr(lay, name)
        assert off % 256 == 0 and off >= end, name      # aligned, in order, no overlap
        end = off + nbytes
    assert lay.bytes >= end and lay.bytes % 256 == 0
    views = api.step_views(torch.zeros(lay.bytes, dtype=torch.uint8),
                           lay, B, nq, H, mp)
    assert views["q"].shape == (T, H, 576) and views["page_table"].shape == (B, mp)
    out = api.StepLayout()
    assert L.dsa_step_layout_get(0, 1, 128, 4, ctypes.byref(out)) == 1
    assert L.dsa_step_layout_get(2, 5, 128, 4, ctypes.byref(out)) == 2
    assert L.dsa_step_layout_get(2, 1, 128, 4, None) == 1


def test_host_step_rejects_bad_arguments_before_any_copy(L):
    d = ctypes.byref(_fake_desc())
    n1 = L.dsa_workspace_bytes(d, 256, 1)
    call = lambda hin, din, ws_bytes, scale=0.07: L.dsa_decode_step_host(
        d, hin, din, FAKE, FAKE, FAKE, scale, 1, 256, FAKE, FAKE, FAKE, ws_bytes, None)
    assert call(None, FAKE, n1) == 1                     # no host block
    assert call(FAKE, None, n1) == 1                     # no device block
    assert call(FAKE, FAKE + 16, n1) == 1                # device block not 256-byte aligned
    assert call(FAKE, FAKE, n1 - 1) == 3                 # short workspace
    assert call(FAKE, FAKE, n1, scale=-1.0) == 1         # bad softmax scale
    assert L.dsa_decode_step_host(ctypes.byref(_fake_desc(q_per_req=5)), FAKE, FAKE, FAKE, FAKE,
                                  FAKE, 0.07, 1, 256, FAKE, FAKE, FAKE, n1, None) == 2


def test_step_ring_rejects_bad_arguments_before_any_copy(L):
    d = _fake_desc()
    r = api.StepRing()
    for b in range(2):
        r.dev_in[b], r.out[b] = FAKE + 0x100000 * b, FAKE + 0x200000 + 0x100000 * b
        r.ev_in[b] = r.ev_done[b] = r.ev_out[b] = 0x1000 + b
    r.ws, r.ws_bytes, r.step = FAKE, 1 << 40, 0
    args = lambda: (ctypes.byref(d), ctypes.byref(r), FAKE, FAKE, FAKE, FAKE, FAKE, 0.07, 0, 256,
                    None)
    assert L.dsa_decode_step_ring(None, ctypes.byref(r), FAKE, FAKE, FAKE, FAKE, FAKE, 0.07, 0,
                                  256, None) == 1
    r.ev_out[1] = None                                    # a missing event
    assert L.dsa_decode_step_ring(*args()) == 1
    r.ev_out[1] = 0x1001
    r.dev_in[0] = FAKE + 16                               # block not 256-byte aligned
    assert L.dsa_decode_step_ring(*args()) == 1
    r.dev_in[0] = FAKE
    assert L.dsa_decode_step_ring(ctypes.byref(_fake_desc(num_heads=100)), ctypes.byref(r), FAKE,
                                  FAKE, FAKE, FAKE, FAKE, 0.07, 0, 256, None) == 2
    r.ws_bytes = 16                                       # workspace too small
    assert L.dsa_decode_step_ring(*args()) == 3
    assert r.step == 0                                    # nothing was queued


def test_mli_validation(L):
    d = ctypes.byref(_fake_desc())
    n1 = L.dsa_workspace_bytes(d, 256, 0)
    call = lambda prev, nxt, q_fp8=FAKE, ws_bytes=n1, splits=0: L.dsa_decode_mli(
        d, q_fp8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, prev, nxt, 0.07, splits, 256, FAKE, FAKE,
        ws_bytes, None)
    assert call(None, FAKE) == 1                 # the selection to attend is required
    assert call(FAKE, None) == 1                 # and the one to write
    assert call(FAKE, FAKE + 2) == 1             # misaligned
    assert call(FAKE, FAKE, q_fp8=None) == 1     # the indexer inputs are required
    assert call(FAKE, FAKE, ws_bytes=16) == 3
    assert call(FAKE, FAKE, splits=33) == 1      # more splits than 64-key tiles
    s = L.dsa_num_splits_mli(d)
    assert 1 <= s <= L.dsa_num_splits_auto(d)
    assert L.dsa_workspace_bytes(d, 256, s) <= n1


def test_merge_validation(L):
    assert L.dsa_merge(-1, 2, FAKE, FAKE, FAKE, None, None) == 1
    assert L.dsa_merge(4, 0, FAKE, FAKE, FAKE, None, None) == 1
    assert L.dsa_merge(4, 33, FAKE, FAKE, FAKE, None, None) == 2
    assert L.dsa_merge(4, 2, FAKE + 4, FAKE, FAKE, None, None) == 1
    assert L.dsa_merge(0, 2, FAKE, FAKE, FAKE, None, None) == 0


def test_package_import_does_not_load_and_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    import deepseek_sparse_attention_lightning_gb300 as pkg
    importlib.reload(pkg)
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        api.lib()


@pytest.mark.parametrize("batch,q_per_req,topk", [(1, 1, 2048), (8, 1, 2048), (4, 1, 2048),
                                                  (32, 2, 2048), (128, 1, 2048), (1024, 1, 64),
                                                  (3, 4, 512), (76, 1, 2048)])
def test_split_rules_stay_in_range(L, batch, q_per_req, topk):
    d = ctypes.byref(_fake_desc(batch=batch, q_per_req=q_per_req, topk=topk, max_pages=4096,
                                num_pages=8192))
    tiles = (topk + 63) // 64
    auto, mli = L.dsa_num_splits_auto(d), L.dsa_num_splits_mli(d)
    assert 1 <= mli <= auto <= tiles
    # the split count divides the positions into equal 64-key-tile blocks with no empty one
    for s in (auto, mli):
        per = -(-tiles // s)
        assert -(-tiles // per) == s
    # a workspace sized for the automatic count also covers the MLI layer's
    assert L.dsa_workspace_bytes(d, 4096 * 64, mli) <= L.dsa_workspace_bytes(d, 4096 * 64, 0)


@pytest.mark.parametrize("batch,q_per_req,heads,max_pages", [(1, 1, 16, 1), (7, 3, 48, 33),
                                                             (1024, 1, 128, 2048), (5, 4, 128, 3)])
def test_step_layout_alignment_across_sizes(L, batch, q_per_req, heads, max_pages):
    lay = api.dsa_step_layout_get(batch, q_per_req, heads, max_pages)
    T = batch * q_per_req
    sizes = [T * 64 * 128, T * 4, T * 64 * 4, T * heads * 576 * 2, batch * 4, batch * max_pages * 4]
    offs = [lay.q_fp8, lay.q_scale, lay.w, lay.q, lay.seqlens, lay.page_table]
    assert all(o % 256 == 0 for o in offs) and lay.bytes % 256 == 0
    ends = [o + n for o, n in zip(offs, sizes)]
    assert all(e <= o for e, o in zip(ends[:-1], offs[1:])) and ends[-1] <= lay.bytes


def _declared_prototypes():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(dsa_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        params = " ".join(m.group(2).split())
        protos[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_binding_signatures_match_the_header():
    protos = _declared_prototypes()
    assert protos, "no prototypes parsed"
    for name, n in protos.items():
        assert name in api._SIGS, f"{name} declared but not bound"
        assert len(api._SIGS[name][1]) == n, f"{name}: header has {n} parameters, binding {len(api._SIGS[name][1])}"
