"""dsa_sparse_decode_attn_noalloc: the split-K sparse attention for callers that cannot allocate.

Callers inside a host framework that owns all device memory, or in loops that cannot accept the
device synchronisation an allocation may cause, cannot hand the library a workspace.  The
no-allocation variant keeps its split records in a fixed device array inside the library.  Here
it is called through the C ABI twice in a row, with different inputs, and with the same explicit
number of splits as the workspace-taking entry point (so both run the split-records path and the
fixed array is really used); each result is checked against that entry point and against the
float64 oracle with the tolerance the other parity tests use.  The file is collected last so that
a failure here never hides the rest of the suite.
"""

import math

import numpy as np
import pytest
import torch

from dynamic_block_sparse_gb300 import binding as B
from dynamic_block_sparse_gb300.pipeline import Cache
from dynamic_block_sparse_gb300.workloads import Workload, make_inputs
from support import assert_outputs, attend_pages, to_cuda

pytestmark = pytest.mark.gpu


def _case(seed):
    w = Workload("noalloc", 2, 32, 2, 128, 64 * 60 + 11, 64, 64, "minmax", "topk", k=40, seed=seed,
                 ragged=True, extra_phys_pages=3)
    inp = to_cuda(make_inputs(w, "cpu"))
    cache = Cache(inp["k_pages"], inp["v_pages"], inp["page_table"], inp["seq_lens"], 32)
    g = np.random.default_rng(seed)
    rows = w.batch * w.num_kv_heads
    idx = np.full((rows, w.k), -1, dtype=np.int32)
    cnt = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        npos = -(-int(inp["seq_lens"][r // 2]) // 64)
        c = min(w.k, npos) - (r % 3)
        idx[r, :c] = np.sort(g.choice(npos, c, replace=False))
        cnt[r] = c
    return w, inp, cache, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()


SPLITS = 8


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    scale = 1 / math.sqrt(128)
    for call, seed in enumerate((3, 4)):
        w, inp, cache, idx, cnt = _case(seed)
        q = inp["q"][0]
        need = B.dsa_sparse_decode_attn_workspace_size(cache.kv, w.k, SPLITS)
        assert need > 0, "the case must use split records"
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = cache.outputs()
        B.dsa_sparse_decode_attn(cache.kv, q, idx, cnt, scale, *ref, num_splits=SPLITS,
                                 workspace=ws)
        got = cache.outputs()
        B.dsa_sparse_decode_attn_noalloc(cache.kv, q, idx, cnt, scale, *got, num_splits=SPLITS)
        torch.cuda.synchronize()
        got_np = [t.cpu().numpy() for t in got]
        assert_outputs(*got_np, [t.double().cpu().numpy() for t in ref], f"no-alloc call {call}")
        # and against the oracle, row by row
        G = w.group
        for b in range(w.batch):
            L = int(inp["seq_lens"][b])
            for h in range(w.num_kv_heads):
                r = b * w.num_kv_heads + h
                pages = idx[r, :int(cnt[r])].cpu().tolist()
                oref = attend_pages(q[b, h * G:(h + 1) * G], inp["k_pages"], inp["v_pages"],
                                    inp["page_table"], L, b, h, pages, scale)
                sl = slice(h * G, (h + 1) * G)
                assert_outputs(got_np[0][b, sl], got_np[1][b, sl], got_np[2][b, sl], oref,
                               f"no-alloc call {call} vs oracle b{b} h{h}")


def test_noalloc_rejects_more_split_records_than_its_scratch():
    w, inp, cache, idx, cnt = _case(5)
    G, rows = w.group, w.batch * w.num_kv_heads
    splits = B.dsa_sparse_decode_attn_noalloc_max_bytes() // (rows * G * 528) + 1
    big = torch.full((w.batch, w.num_kv_heads, splits), 0, dtype=torch.int32, device="cuda")
    out, m, l = cache.outputs()
    with pytest.raises(B.DsaError, match="scratch"):
        B.dsa_sparse_decode_attn_noalloc(cache.kv, inp["q"][0], big, cnt, 0.1, out, m, l,
                                         num_splits=splits)
