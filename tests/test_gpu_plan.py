"""The split planner's output, read back from the workspace, is a valid
work split: every page of every sequence is taken by exactly one worker, in
order; each sequence's split count, first worker and partial slots agree
with the workers' ranges; and no worker's cost (pages plus the per-sequence
fixed cost the plan assumes) exceeds the per-worker share by more than one
sequence's fixed cost. Record layouts follow csrc/common.cuh."""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth

pytestmark = pytest.mark.gpu

PAGE = 64
C_SEG_TC = 4  # fixed cost units per sequence the tcgen05 plan charges


def align(v, a):
    return (v + a - 1) // a * a


def plan(lens, max_pages):
    wl = synth.WORKLOADS["dsv2_b32_ctx4k"]
    dims = M.Dims.of(wl)
    B = len(lens)
    ws = torch.zeros(M.mla_decode_workspace_size(B, M.MLA_BF16, dims), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_plan_decode(torch.tensor(lens, dtype=torch.int32, device="cuda"), max_pages, ws,
                      M.MLA_BF16, dims, status)
    torch.cuda.synchronize()
    raw = ws.cpu().numpy().view(np.int32)
    hdr = raw[:8]
    workers = int(hdr[0])
    seqs = raw[256 // 4:256 // 4 + 8 * B].reshape(B, 8)
    w0 = align(256 + 32 * B, 256) // 4
    wk = raw[w0:w0 + 8 * workers].reshape(workers, 8)
    return hdr, seqs, wk, int(status.item()), M.mla_decode_path(M.MLA_BF16, dims)


def check(lens, max_pages):
    hdr, seqs, wk, status, path = plan(lens, max_pages)
    workers, per, total, num_slots, batch = (int(x) for x in hdr[:5])
    B = len(lens)
    assert batch == B
    assert int(hdr[5]) == path
    assert int(hdr[6]) == 1  # a bf16 cache keeps its split partials in bf16
    valid = [1 <= n <= max_pages * PAGE for n in lens]
    assert (status != 0) == (not all(valid))
    pages = [(n + PAGE - 1) // PAGE if ok else 0 for n, ok in zip(lens, valid)]
    assert list(seqs[:, 1]) == pages
    assert total == sum(pages)
    # every worker's (sequence, page) range, in worker order
    owner = {}
    order = []
    costs = []
    for g in range(workers):
        sb, pb, se, pe, n = (int(x) for x in wk[g, :5])
        if n == 0:
            costs.append(0)
            continue
        got, segs = [], 0
        for s in range(sb, se + 1):
            p0 = pb if s == sb else 0
            p1 = pe + 1 if s == se else pages[s]
            if p1 > p0:
                segs += 1
            for p in range(p0, p1):
                got.append((s, p))
                assert (s, p) not in owner, f"page {(s, p)} taken twice"
                owner[(s, p)] = g
        assert len(got) == n, f"worker {g}: n_pages {n} != {len(got)}"
        order += got
        c = C_SEG_TC if path >= 1 else 0
        costs.append(len(got) + c * segs)
    want = [(s, p) for s in range(B) for p in range(pages[s])]
    assert order == want, "pages not covered exactly once, in order"
    c = C_SEG_TC if path >= 1 else 0
    assert max(costs) <= per + c, f"worker cost {max(costs)} > per {per} + {c}"
    # per-sequence split records and partial slots
    slot = 0
    for s in range(B):
        ws_ = sorted({owner[(s, p)] for p in range(pages[s])})
        n_splits, first, slot_begin = int(seqs[s, 3]), int(seqs[s, 2]), int(seqs[s, 4])
        assert n_splits == len(ws_), f"seq {s}: n_splits {n_splits} != {len(ws_)}"
        if ws_:
            assert first == ws_[0] and ws_ == list(range(ws_[0], ws_[0] + len(ws_)))
        if n_splits > 1:
            assert slot_begin == slot
            slot += n_splits
    assert num_slots == slot


@pytest.mark.parametrize("name", ["dsv2_b32_ctx4k", "dsv2_b4_ctx128k", "dsv2_b128_ragged"])
def test_plan_of_the_workloads(name):
    wl = synth.WORKLOADS[name]
    lens = synth.seq_lens(wl)
    check([int(x) for x in lens], int((lens.max() + PAGE - 1) // PAGE))


def test_plan_edge_cases():
    check([1], 1)                                   # one token
    check([64, 65, 1, 128], 2)                      # page boundaries
    check([0, 100, 4096, -5, 10 ** 6], 64)          # invalid lengths among valid ones
    check([7] * 300, 1)                             # many one-page sequences
    check([131072, 1, 131072], 2048)                # long ones around a short one


def test_plan_many_sequences_global_path():
    """More sequences than the planner keeps in shared memory (4096)."""
    rng = np.random.default_rng(67011)
    lens = [int(x) for x in rng.integers(1, 400, size=5000)]
    check(lens, 7)
