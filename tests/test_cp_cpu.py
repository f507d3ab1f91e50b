"""Context-parallel decode (deepseek_sparse_attention_lightning_gb300.cp) on CPU.

The exchange logic -- local top-k candidates, their all-gather, the global
top-k, the attention over each rank's own winners and the merge of the ranks'
partials -- runs here on gloo ranks (2 and 3 processes), with the per-rank
steps taken by the float64 oracle (test infrastructure), and must give the
single-pass layer of the oracle on the whole request: the same selection and
the same output.  The GPU steps are checked in test_gpu_parity.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_slice_bounds_are_page_aligned_and_cover_the_request():
    from deepseek_sparse_attention_lightning_gb300 import cp
    for S in (1, 63, 64, 65, 700, 4096, 131072, 131071):
        for R in (1, 2, 3, 8):
            b = cp.slice_bounds(S, R)
            assert b[0] == 0 and b[-1] == S and len(b) == R + 1
            assert all(b[i] <= b[i + 1] for i in range(R))
            assert all(x % 64 == 0 for x in b[:-1])
    assert cp.slice_bounds(4096, 4) == [0, 1024, 2048, 3072, 4096]


class OracleSteps:
    """The per-rank steps taken by the oracle on this rank's slice (the
    global caches viewed through the slice's page table)."""

    def __init__(self, a, bounds_r, k):
        import oracle as O
        self.O, self.a, self.k = O, a, k
        B = a["seqlens"].shape[0]
        self.len = np.array([hi - lo for lo, hi in bounds_r], dtype=np.int64)
        mp_ = max(1, int(max((n + 63) // 64 for n in self.len)))
        self.table = np.full((B, mp_), -1, dtype=np.int64)
        for i, (lo, hi) in enumerate(bounds_r):
            npg = (hi - lo + 63) // 64
            self.table[i, :npg] = a["page_table"][i, lo // 64: lo // 64 + npg]
        self.ld = mp_ * 64

    def scores(self):
        a, O = self.a, self.O
        I, _ = O.indexer_logits(a["q_fp8"], a["q_scale"], a["w"], a["k_fp8"], a["k_scale"],
                                self.table, self.len, 1, with_bound=False)
        out = np.full((I.shape[0], self.ld), -np.inf, dtype=np.float32)
        out[:, :I.shape[1]] = I.astype(np.float32)
        return torch.from_numpy(out)

    def local_topk(self, logits):
        return torch.from_numpy(self.O.topk(logits.numpy(), self.len, self.k)).int()

    def global_topk(self, cand_scores):
        n = cand_scores.shape[1]
        vis = np.full(cand_scores.shape[0], n)
        return torch.from_numpy(self.O.topk(cand_scores.numpy(), vis, self.k)).int()

    def attention(self, idx_local):
        a, O = self.a, self.O
        mo, ml = O.sparse_mla_split(a["q"], a["kv"], idx_local.numpy(), self.table, self.len, 1,
                                    a["sm_scale"], 1)
        return torch.from_numpy(mo[:, :, 0]), torch.from_numpy(ml[:, :, 0])

    def merge(self, mid_o, mid_lse):
        o, _ = self.O.merge(mid_o.numpy(), mid_lse.numpy())
        return torch.from_numpy(o)


def _case():
    from deepseek_sparse_attention_lightning_gb300 import workloads as W
    spec = W.small_spec("long_varlen", batch=2, q_per_req=1, num_heads=16, topk=96,
                        heavy="runs:0.05:3", seed=41)
    wl = W.make_workload(spec, seqlens=[1000, 650])
    return W.host_arrays(wl)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from deepseek_sparse_attention_lightning_gb300 import cp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        a = _case()
        bounds = [cp.slice_bounds(int(S), world) for S in a["seqlens"]]
        mine = [(b[rank], b[rank + 1]) for b in bounds]
        sl = cp.RankSlice(start=[lo for lo, _ in mine], length=[hi - lo for lo, hi in mine])
        o, sel = cp.run_distributed(OracleSteps(a, mine, a["topk"]), sl)
        out.put((rank, o.numpy(), sel.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_layer_equals_single_pass(world):
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    a = _case()
    want = O.decode_layer(a)
    for _, o, sel in res:
        assert np.array_equal(sel, want["idx"])           # the global selection, every rank
        assert np.allclose(o, want["out"], rtol=1e-9, atol=1e-12)
