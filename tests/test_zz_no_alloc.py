"""dsa_topk_noalloc: the top-k entry point for callers that cannot allocate.

Some callers run the selection where no device allocation is allowed (an
engine step that already handed all device memory to its caches, a runtime
without its own device allocator).  dsa_topk_noalloc keeps its scratch in a
fixed device array inside the library instead of taking a workspace.  This
test calls it through the C ABI and checks that it selects exactly what
dsa_topk (the workspace version) selects, on two calls in a row, so that the
second call cannot lean on state the first one left behind.  The file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from deepseek_sparse_attention_lightning_gb300 import api


def _desc(vis_rows, ld, k):
    seqlens = torch.tensor(vis_rows, dtype=torch.int32, device="cuda")
    table = torch.zeros((len(vis_rows), ld // 64), dtype=torch.int32, device="cuda")
    return api.make_desc(seqlens, table, 1, 128, k, ld // 64), (seqlens, table)


def _both(scores, vis_rows, k):
    T, ld = scores.shape
    desc, keep = _desc(vis_rows, ld, k)
    logits = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    ref = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(api.dsa_topk_workspace_bytes(desc, ld), dtype=torch.uint8, device="cuda")
    api.dsa_topk(desc, logits, ref, ws, ld)
    got = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    api.dsa_topk_noalloc(desc, logits, got, ld)
    torch.cuda.synchronize()
    assert api.dsa_get_device_error() == 0
    return got.cpu().numpy(), ref.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_topk_matches_workspace_topk_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_sparse_attention_lightning_gb300 import build
    build.build()
    rng = np.random.default_rng(77)
    # call 1: 16 rows x 131072 scores (T * ld = 2^21, the limit), k = 2048
    s1 = rng.standard_normal((16, 131072)).astype(np.float32)
    vis1 = [131072 - 3 * i for i in range(16)]
    got, ref = _both(s1, vis1, 2048)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, O.topk(s1, vis1, 2048))
    # call 2 right after: other shapes, many ties and short rows; the scratch
    # still holds call 1's histogram and counters
    s2 = (np.round(rng.standard_normal((40, 8192)) * 2) / 2).astype(np.float32)
    vis = [8192 - 5 * i for i in range(38)] + [100, 2048]
    got, ref = _both(s2, vis, 512)
    assert np.array_equal(got, ref)
    assert np.array_equal(got, O.topk(s2, vis, 512))


@pytest.mark.gpu
def test_noalloc_topk_back_to_back_on_one_stream():
    """Two calls of different shapes queued on one non-default stream with no
    host synchronisation between them: the second call's clearing of the
    shared scratch is ordered after the first call's kernels by the stream,
    so both selections must still equal dsa_topk's and the oracle's."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deepseek_sparse_attention_lightning_gb300 import build
    build.build()
    rng = np.random.default_rng(78)
    cases = [(rng.standard_normal((8, 65536)).astype(np.float32), [65536 - 7 * i for i in range(8)], 2048),
             ((np.round(rng.standard_normal((24, 16384)) * 4) / 4).astype(np.float32),
              [16384 - 11 * i for i in range(23)] + [700], 1024)]
    stream = torch.cuda.Stream()
    keep, outs = [], []
    with torch.cuda.stream(stream):
        for scores, vis, k in cases:
            T, ld = scores.shape
            desc, bufs = _desc(vis, ld, k)
            logits = torch.from_numpy(scores).to("cuda", non_blocking=False)
            got = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
            keep.append((desc, bufs, logits))
            outs.append(got)
    stream.synchronize()
    for (desc, _, logits), got in zip(keep, outs):
        api.dsa_topk_noalloc(desc, logits, got, int(logits.shape[1]), stream=stream)
    stream.synchronize()
    assert api.dsa_get_device_error() == 0
    for (scores, vis, k), (desc, _, logits), got in zip(cases, keep, outs):
        ld = int(logits.shape[1])
        ref = torch.full_like(got, -7)
        ws = torch.empty(api.dsa_topk_workspace_bytes(desc, ld), dtype=torch.uint8, device="cuda")
        api.dsa_topk(desc, logits, ref, ws, ld)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy())
        assert np.array_equal(got.cpu().numpy(), O.topk(scores, vis, k))


def test_noalloc_topk_rejects_sizes_beyond_its_scratch():
    # host-side check: returns before touching the GPU
    build = pytest.importorskip("deepseek_sparse_attention_lightning_gb300.build")
    build.build()
    L = api.lib()
    FAKE = 0x7f0000000000
    d = api.DecodeDesc(batch=65, q_per_req=1, num_heads=128, topk=2048, page_size=64, max_pages=4,
                       num_pages=8, seqlens=0x10000, page_table=0x20000)
    assert L.dsa_topk_noalloc(ctypes.byref(d), FAKE, 256, FAKE, None) == 2     # T > 64
    d.batch = 32
    d.max_pages = 2048
    assert L.dsa_topk_noalloc(ctypes.byref(d), FAKE, 131072, FAKE, None) == 2  # T*ld > 2^21


def test_noalloc_topk_rejects_what_dsa_topk_rejects():
    # host-side: the descriptor checks are shared, so both entry points return
    # the same status for the same bad descriptor
    build = pytest.importorskip("deepseek_sparse_attention_lightning_gb300.build")
    build.build()
    L = api.lib()
    FAKE = 0x7f0000000000
    ws = 1 << 30
    base = dict(batch=2, q_per_req=1, num_heads=128, topk=2048, page_size=64, max_pages=4,
                num_pages=8, seqlens=0x10000, page_table=0x20000)
    for over, want in [(dict(num_heads=20), 2), (dict(num_heads=256), 2),
                       (dict(num_pages=1 << 26), 2), (dict(page_size=32), 2),
                       (dict(batch=0), 1), (dict(seqlens=0x10002), 1), (dict(topk=0), 1)]:
        d = api.DecodeDesc(**{**base, **over})
        a = L.dsa_topk_noalloc(ctypes.byref(d), FAKE, 256, FAKE, None)
        b = L.dsa_topk(ctypes.byref(d), FAKE, 256, FAKE, FAKE, ws, None)
        assert a == b == want, (over, a, b)
