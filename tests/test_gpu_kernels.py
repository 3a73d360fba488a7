"""Kernel-by-kernel parity of libdsa against the float64 oracle (one C-ABI call per test)."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from dynamic_block_sparse_gb300 import binding as B
from dynamic_block_sparse_gb300.pipeline import Cache
from dynamic_block_sparse_gb300.workloads import Workload, make_inputs
from support import (assert_outputs, attend_pages, check_topk, f64, oracle_mean_scores,
                     oracle_minmax_scores, row_tokens, to_cuda)

pytestmark = pytest.mark.gpu


def small(B_=2, Hq=8, Hkv=2, L=700, page=16, lp=None, kind="minmax", extra=5, seed=7, hot=0,
          streaming=()):
    w = Workload("unit", B_, Hq, Hkv, 128, L, page, lp or page, kind, "topk", k=8, hot_pages=hot,
                 hot_scale=0.5, seed=seed, ragged=True, extra_phys_pages=extra,
                 streaming_kv_heads=streaming)
    inp = to_cuda(make_inputs(w, "cpu"))
    cache = Cache(inp["k_pages"], inp["v_pages"], inp["page_table"], inp["seq_lens"], Hq,
                  inp["head_is_streaming"] if streaming else None)
    return w, inp, cache


def keys_values(inp, cache, b, h):
    L = int(inp["seq_lens"][b])
    return (row_tokens(inp["k_pages"], inp["page_table"], L, b, h),
            row_tokens(inp["v_pages"], inp["page_table"], L, b, h), L)


# ---------------------------------------------------------------------------------- metadata

@pytest.mark.parametrize("page,lp", [(16, 16), (64, 16), (64, 64), (32, 8)])
@pytest.mark.parametrize("kind", ["minmax", "mean"])
def test_build_page_meta(page, lp, kind):
    w, inp, cache = small(page=page, lp=lp, kind=kind, L=page * 9 + 5)
    code = B.DSA_META_MINMAX if kind == "minmax" else B.DSA_META_MEAN
    meta = cache.meta_buffer(code, lp)
    B.dsa_build_page_meta(cache.kv, code, lp, meta)
    torch.cuda.synchronize()
    g = page // lp
    table = inp["page_table"].cpu().numpy()
    mcpu = meta.float().cpu().numpy()
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            K, _, L = keys_values(inp, cache, b, h)
            if kind == "minmax":
                kmax, kmin = O.page_meta_minmax(K, lp)
                for j in range(len(kmax)):
                    rec = mcpu[table[b, j // g], h, j % g]
                    np.testing.assert_array_equal(rec[:, 0], kmax[j])
                    np.testing.assert_array_equal(rec[:, 1], kmin[j])
            else:
                mean = O.page_meta_mean(K, lp)
                for j in range(len(mean)):
                    rec = mcpu[table[b, j // g], h, j % g]
                    np.testing.assert_allclose(rec, mean[j], rtol=1e-6, atol=1e-6)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("page,lp,kind", [(16, 16, "minmax"), (64, 16, "minmax"),
                                          (32, 8, "mean"), (64, 64, "mean")])
def test_append_kv_keeps_metadata_exact(page, lp, kind):
    """Decode-time KV append (LServe §4.2): each request loses 2 pages + 3 tokens of its context,
    then grows back one token at a time (crossing page boundaries) with fresh random K/V.  After
    every append the pools hold the token and the incrementally kept metadata equals a full
    rebuild bit for bit; at the end it also equals the oracle's metadata of the grown context."""
    w, inp, cache = small(page=page, lp=lp, kind=kind, L=page * 9 + 5)
    code = B.DSA_META_MINMAX if kind == "minmax" else B.DSA_META_MEAN
    grow = 2 * page + 3
    L_end = cache.seq_lens.clone()
    cache.seq_lens.sub_(torch.clamp(L_end - 1, max=grow))      # every request keeps >= 1 token
    meta = cache.meta_buffer(code, lp)
    B.dsa_build_page_meta(cache.kv, code, lp, meta)
    gen = torch.Generator(device="cuda").manual_seed(21)
    kp, vp = cache.k_pages.clone(), cache.v_pages.clone()     # the expected pools
    table = cache.page_table.long()
    for step in range(grow):
        live = cache.seq_lens < L_end
        if not bool(live.any()):
            break
        k_new = torch.randn((w.batch, w.num_kv_heads, 128), generator=gen, device="cuda")
        v_new = torch.randn((w.batch, w.num_kv_heads, 128), generator=gen, device="cuda")
        k_new, v_new = k_new.bfloat16(), v_new.bfloat16()
        # requests that reached their length append nothing: their length stays 0-advanced
        lens = cache.seq_lens + live.int()
        cache.seq_lens.copy_(lens)
        for b in range(w.batch):
            if not bool(live[b]):
                continue
            t = int(lens[b]) - 1
            phys = int(table[b, t // page])
            kp[phys, :, t % page] = k_new[b]
            vp[phys, :, t % page] = v_new[b]
        # a request that did not grow is given its current last token again (a no-op rewrite)
        for b in range(w.batch):
            if not bool(live[b]):
                t = int(lens[b]) - 1
                phys = int(table[b, t // page])
                k_new[b] = kp[phys, :, t % page]
                v_new[b] = vp[phys, :, t % page]
        B.dsa_append_kv(cache.kv, k_new, v_new, code, lp, meta)
        full = cache.meta_buffer(code, lp)
        B.dsa_build_page_meta(cache.kv, code, lp, full)
        torch.cuda.synchronize()
        assert torch.equal(cache.k_pages, kp) and torch.equal(cache.v_pages, vp), f"pools {step}"
        assert torch.equal(meta, full), f"metadata after append {step}"
    assert torch.equal(cache.seq_lens, L_end)
    g = page // lp
    mcpu = meta.float().cpu().numpy()
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            L = int(L_end[b])
            K = row_tokens(cache.k_pages, cache.page_table, L, b, h)
            if kind == "minmax":
                kmax, kmin = O.page_meta_minmax(K, lp)
                for jj in range(len(kmax)):
                    rec = mcpu[int(table[b, jj // g]), h, jj % g]
                    np.testing.assert_array_equal(rec[:, 0], kmax[jj])
                    np.testing.assert_array_equal(rec[:, 1], kmin[jj])
            else:
                mean = O.page_meta_mean(K, lp)
                for jj in range(len(mean)):
                    rec = mcpu[int(table[b, jj // g]), h, jj % g]
                    np.testing.assert_allclose(rec, mean[jj], rtol=1e-6, atol=1e-6)
    assert int(cache.status.item()) == 0


def test_decode_loop_with_kv_append():
    """A top-K decode loop that appends each step's token before attending (the metadata kept by
    the appends, never rebuilt): every step selects the oracle's top-K over the grown context and
    attends exactly over it."""
    w, inp, cache = small(page=16, L=16 * 40 + 9, seed=8)
    grow = 20
    L_end = cache.seq_lens.clone()
    cache.seq_lens.sub_(grow)
    from dynamic_block_sparse_gb300.pipeline import TopKDecoder
    dec = TopKDecoder(cache, 12)
    dec.build_meta()
    gen = torch.Generator(device="cuda").manual_seed(22)
    G = w.num_q_heads // w.num_kv_heads
    for step in range(grow):
        k_new = torch.randn((w.batch, w.num_kv_heads, 128), generator=gen, device="cuda").bfloat16()
        v_new = torch.randn((w.batch, w.num_kv_heads, 128), generator=gen, device="cuda").bfloat16()
        q = torch.randn((w.batch, w.num_q_heads, 128), generator=gen, device="cuda").bfloat16()
        dec.append(k_new, v_new)
        out, m, l = dec.step(q)
        torch.cuda.synchronize()
        if step % 5 != 4:
            continue
        for b in range(w.batch):
            L = int(cache.seq_lens[b])
            for h in range(w.num_kv_heads):
                K = row_tokens(cache.k_pages, cache.page_table, L, b, h)
                qg = q[b, h * G:(h + 1) * G]
                IS = oracle_minmax_scores(K, qg, 16, dec.stride)
                A = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
                check_topk(A, IS, 12, f"step {step} b{b} h{h}")
                ref = attend_pages(qg, cache.k_pages, cache.v_pages, cache.page_table, L, b, h,
                                   sorted(A.tolist()), dec.scale)
                sl = slice(h * G, (h + 1) * G)
                assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(),
                               l[b, sl].cpu().numpy(), ref, f"step {step} b{b} h{h}")
    assert torch.equal(cache.seq_lens, L_end)
    assert int(cache.status.item()) == 0


# ---------------------------------------------------------------------------------- scoring

@pytest.mark.parametrize("page,lp,Hq,Hkv", [(16, 16, 8, 2), (64, 16, 16, 4), (64, 64, 32, 2),
                                           (16, 16, 4, 4)])
@pytest.mark.parametrize("kind", ["minmax", "mean"])
def test_score_pages(page, lp, Hq, Hkv, kind):
    w, inp, cache = small(Hq=Hq, Hkv=Hkv, page=page, lp=lp, kind=kind, L=page * 23 + 3,
                          streaming=(1,) if Hkv > 2 else ())
    code = B.DSA_META_MINMAX if kind == "minmax" else B.DSA_META_MEAN
    meta = cache.meta_buffer(code, lp)
    B.dsa_build_page_meta(cache.kv, code, lp, meta)
    stride = cache.max_pages * (page // lp) + 3
    scores = torch.full((w.batch, Hkv, stride), 7.0, device="cuda")
    q = inp["q"][0]
    B.dsa_score_pages(cache.kv, q, meta, code, lp, scores)
    s = scores.double().cpu().numpy()
    G = Hq // Hkv
    for b in range(w.batch):
        for h in range(Hkv):
            if h in w.streaming_kv_heads:
                assert np.all(np.isneginf(s[b, h]))
                continue
            K, _, L = keys_values(inp, cache, b, h)
            qg = q[b, h * G:(h + 1) * G]
            ref = (oracle_minmax_scores if kind == "minmax" else oracle_mean_scores)(K, qg, lp, stride)
            nl = -(-L // lp)
            assert np.all(np.isneginf(s[b, h, nl:]))
            scale = np.abs(ref[:nl]).max()
            np.testing.assert_allclose(s[b, h, :nl], ref[:nl], rtol=1e-5, atol=1e-6 * scale)


# ---------------------------------------------------------------------------------- selection

def _tied_scores(rows, n, seed, neg_inf_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    s = torch.round(torch.randn(rows, n, generator=g) * 4) / 4       # many exact ties
    s[torch.rand(rows, n, generator=g) < neg_inf_frac] = -math.inf
    s[0, : min(n, 3)] = torch.tensor([0.0, -0.0, 0.0])[: min(n, 3)]   # signed zeros tie
    if rows > 1:
        s[1] = -math.inf                                               # a row with nothing valid
    return s


@pytest.mark.parametrize("n,k", [(1, 1), (37, 5), (37, 0), (2048, 256), (8192, 64), (8192, 76),
                                 (32768, 1000), (300, 400)])
def test_select_topk_exact(n, k):
    s = _tied_scores(5, n, seed=n + k)
    stride = n + 3
    sd = torch.full((5, stride), -math.inf)
    sd[:, :n] = s
    sd = sd.cuda()
    idx = torch.full((5, max(k, 1)), -7, dtype=torch.int32, device="cuda")
    cnt = torch.empty(5, dtype=torch.int32, device="cuda")
    B.dsa_select_topk(sd, n, k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(5):
        ref = O.select_topk(s[r].double().numpy(), k)
        assert cnt[r] == len(ref)
        assert list(idx[r, :cnt[r]]) == ref
        assert np.all(idx[r, cnt[r]:k] == -1)


def test_select_topk_crowded_cutoff():
    """Rows whose cut-off bin holds more keys than the one-pass path gathers (all keys equal; 600
    keys tied at the k-th score; two values only) take the radix path and give the same exact
    selection; rows with a few keys per bin take the one-pass path."""
    n, k = 8192, 64
    g = torch.Generator().manual_seed(5)
    rows = [torch.ones(n), torch.randn(n, generator=g), torch.where(torch.rand(n, generator=g) < 0.5,
                                                                    1.0, 2.0)]
    r = torch.randn(n, generator=g) - 10.0
    r[torch.randperm(n, generator=g)[:600]] = 3.0
    r[torch.randperm(n, generator=g)[:20]] = 7.0
    rows.append(r)
    s = torch.stack(rows)
    idx = torch.full((len(rows), k), -7, dtype=torch.int32, device="cuda")
    cnt = torch.empty(len(rows), dtype=torch.int32, device="cuda")
    B.dsa_select_topk(s.cuda(), n, k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for i in range(len(rows)):
        ref = O.select_topk(s[i].double().numpy(), k)
        assert cnt[i] == k and list(idx[i]) == ref, f"row {i}"


@pytest.mark.parametrize("n_logical,g,k", [(8192, 4, 64), (1001, 4, 12), (64, 1, 8), (999, 3, 50)])
def test_select_hier_exact(n_logical, g, k):
    s = _tied_scores(4, n_logical, seed=g * 100 + k)
    sd = s.cuda()
    idx = torch.empty((4, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty(4, dtype=torch.int32, device="cuda")
    B.dsa_select_hier(sd, n_logical, g, k, idx, cnt)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for r in range(4):
        ref = O.select_hier(s[r].double().numpy(), g, k)
        assert list(idx[r, :cnt[r]]) == ref


# ---------------------------------------------------------------------------------- attention

def _random_selection(w, inp, k, seed, allow_bad=True):
    g = np.random.default_rng(seed)
    rows = w.batch * w.num_kv_heads
    idx = np.full((rows, k), -1, dtype=np.int32)
    cnt = np.zeros(rows, dtype=np.int32)
    for r in range(rows):
        b = r // w.num_kv_heads
        npos = -(-int(inp["seq_lens"][b]) // w.page_size)
        c = int(g.integers(0, min(k, npos) + 1)) if r % 3 else min(k, npos)
        sel = sorted(g.choice(npos, c, replace=False).tolist())
        if allow_bad and r == 1 and c > 0:
            sel[-1] = npos + 3                                  # out of range: skipped
        idx[r, :c] = sel
        cnt[r] = c
    return idx, cnt


def _oracle_sparse(w, inp, cache, q, idx, cnt, scale):
    G = w.group
    O_ref = np.zeros((w.batch, w.num_q_heads, 128))
    m_ref = np.full((w.batch, w.num_q_heads), -np.inf)
    l_ref = np.zeros((w.batch, w.num_q_heads))
    for r in range(idx.shape[0]):
        b, h = divmod(r, w.num_kv_heads)
        K, V, L = keys_values(inp, cache, b, h)
        npos = -(-L // w.page_size)
        pages = [int(j) for j in idx[r, :cnt[r]] if 0 <= j < npos]
        res = O.attend(q[b, h * G:(h + 1) * G], K, V, O.page_token_ids(pages, w.page_size, L), scale)
        O_ref[b, h * G:(h + 1) * G], m_ref[b, h * G:(h + 1) * G], l_ref[b, h * G:(h + 1) * G] = res
    return O_ref, m_ref, l_ref


@pytest.mark.parametrize("Hq,Hkv,page", [(8, 2, 16), (4, 4, 16), (32, 2, 64), (16, 2, 32),
                                         (24, 2, 16)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_sparse_decode_attn(Hq, Hkv, page, splits):
    w, inp, cache = small(Hq=Hq, Hkv=Hkv, page=page, L=page * 40 + 9, seed=Hq + page)
    k = 24
    idx, cnt = _random_selection(w, inp, k, seed=splits + Hq)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    ws = B.dsa_sparse_decode_attn_workspace_size(cache.kv, k, splits)
    wsb = torch.zeros(max(ws, 16), dtype=torch.uint8, device="cuda")
    out, m, l = cache.outputs()
    B.dsa_sparse_decode_attn(cache.kv, q, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda(),
                             scale, out, m, l, num_splits=splits, workspace=wsb)
    torch.cuda.synchronize()
    ref = _oracle_sparse(w, inp, cache, q, idx, cnt, scale)
    assert_outputs(out.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(), ref, "sparse attn")
    assert int(cache.status.item()) == 0


# The default (persistent) path cuts the global page-slot space into one equal range per CTA:
# one long row split across every CTA, many short rows inside single CTAs, fewer slots than CTAs,
# streaming heads left out of the slot space, and a second call on the same workspace (the row
# tickets must be back at zero).
@pytest.mark.parametrize("shape", ["one_long_row", "many_short_rows", "fewer_slots_than_ctas",
                                   "streaming_heads"])
def test_persistent_partition(shape):
    streaming = ()
    if shape == "one_long_row":
        w, inp, cache = small(B_=1, Hq=8, Hkv=1, page=16, L=16 * 1100 + 3, seed=11)
        k = 1024
    elif shape == "many_short_rows":
        w, inp, cache = small(B_=40, Hq=32, Hkv=8, page=16, L=16 * 30 + 5, seed=12)
        k = 3
    elif shape == "fewer_slots_than_ctas":
        w, inp, cache = small(B_=1, Hq=8, Hkv=2, page=16, L=16 * 9, seed=13)
        k = 5
    else:
        streaming = (1, 3)
        w, inp, cache = small(B_=3, Hq=16, Hkv=4, page=64, L=64 * 50 + 3, seed=14,
                              streaming=streaming)
        k = 20
    idx, cnt = _random_selection(w, inp, k, seed=k, allow_bad=False)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    ws = torch.zeros(max(16, B.dsa_sparse_decode_attn_workspace_size(cache.kv, k)),
                     dtype=torch.uint8, device="cuda")
    ref = _oracle_sparse(w, inp, cache, q, idx, cnt, scale)
    dense = np.array([h not in streaming for h in range(w.num_kv_heads)]).repeat(w.group)
    for call in range(2):
        out, m, l = cache.outputs()
        B.dsa_sparse_decode_attn(cache.kv, q, torch.from_numpy(idx).cuda(),
                                 torch.from_numpy(cnt).cuda(), scale, out, m, l, workspace=ws)
        torch.cuda.synchronize()
        assert_outputs(out.cpu().numpy()[:, dense], m.cpu().numpy()[:, dense],
                       l.cpu().numpy()[:, dense], [x[:, dense] for x in ref],
                       f"{shape} call {call}")
        if streaming:  # rows of streaming heads are not this call's to write
            assert not out[:, ~torch.from_numpy(dense).cuda()].any()
        assert int(cache.status.item()) == 0


@pytest.mark.parametrize("Hq,Hkv,page", [(32, 2, 64), (8, 2, 16)])
def test_page_partials_and_merge(Hq, Hkv, page):
    w, inp, cache = small(Hq=Hq, Hkv=Hkv, page=page, L=page * 30 + 1, seed=3)
    k = 12
    idx, cnt = _random_selection(w, inp, k, seed=5, allow_bad=False)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    G = w.group
    part = torch.full((w.batch, Hkv, k, G, B.RECORD_FLOATS), 9.0, device="cuda")
    out, m, l = cache.outputs()
    B.dsa_sparse_decode_attn(cache.kv, q, torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda(),
                             scale, out, m, l, page_partials=part)
    torch.cuda.synchronize()
    pc = part.cpu().numpy()
    for r in range(w.batch * Hkv):
        b, h = divmod(r, Hkv)
        K, V, L = keys_values(inp, cache, b, h)
        for i in range(cnt[r]):
            ref = O.attend(q[b, h * G:(h + 1) * G], K, V,
                           O.page_token_ids([idx[r, i]], page, L), scale)
            rec = pc[b, h, i]
            assert_outputs(rec[:, :128], rec[:, 128], rec[:, 129], ref, f"record {r},{i}")
    ref = _oracle_sparse(w, inp, cache, q, idx, cnt, scale)
    assert_outputs(out.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy(), ref, "merged partials")


def test_merge_partials_generic():
    g = np.random.default_rng(4)
    rows, parts, G = 3, 5, 4
    rec = np.zeros((rows, parts, G, B.RECORD_FLOATS), dtype=np.float32)
    rec[..., :128] = g.normal(size=(rows, parts, G, 128))
    rec[..., 128] = g.normal(size=(rows, parts, G)) * 3
    rec[..., 129] = g.uniform(0.5, 20, size=(rows, parts, G))
    rec[1, 2, :, 129] = 0.0                  # empty part: identity
    rec[1, 2, :, 128] = -np.inf
    t = torch.from_numpy(rec).cuda()
    out = torch.empty((rows * G, 128), device="cuda")
    m = torch.empty(rows * G, device="cuda")
    l = torch.empty_like(m)
    B.dsa_merge_partials(t, out, m, l)
    for r in range(rows):
        ref = O.merge_partials([(rec[r, p, :, :128].astype(np.float64), rec[r, p, :, 128].astype(np.float64),
                                 rec[r, p, :, 129].astype(np.float64)) for p in range(parts)])
        assert_outputs(out[r * G:(r + 1) * G].cpu().numpy(), m[r * G:(r + 1) * G].cpu().numpy(),
                       l[r * G:(r + 1) * G].cpu().numpy(), ref, f"merge row {r}")


@pytest.mark.parametrize("L,sink,local,page", [(5000, 64, 256, 64), (300, 64, 256, 64),
                                               (200, 64, 256, 16), (1000, 0, 100, 16),
                                               (1000, 50, 0, 16), (4100, 64, 256, 16)])
def test_streaming_head_attn(L, sink, local, page):
    w, inp, cache = small(Hq=16, Hkv=4, page=page, L=L, streaming=(2, 3), seed=L)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    out, m, l = cache.outputs()
    out.fill_(5.0)
    B.dsa_streaming_head_attn(cache.kv, q, sink, local, scale, out, m, l)
    torch.cuda.synchronize()
    G = w.group
    oc, mc, lc = out.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()
    for b in range(w.batch):
        for h in range(4):
            sl = slice(h * G, (h + 1) * G)
            if h not in (2, 3):
                assert np.all(oc[b, sl] == 5.0)          # dense heads untouched
                continue
            K, V, Lb = keys_values(inp, cache, b, h)
            ref = O.attend(q[b, sl], K, V, O.streaming_token_ids(Lb, sink, local), scale)
            assert_outputs(oc[b, sl], mc[b, sl], lc[b, sl], ref, f"stream b{b} h{h}")


@pytest.mark.parametrize("L,sink,local,page", [(16 * 50 + 7, 64, 256, 16), (64 * 30 + 9, 64, 256, 64),
                                               (300, 64, 256, 64), (100, 64, 256, 16),
                                               (64 * 20, 0, 200, 64), (64 * 20 + 3, 40, 0, 64)])
def test_hybrid_decode_attn(L, sink, local, page):
    """Dense and streaming heads in one launch: the dense heads attend exactly their selected pages
    and the streaming heads exactly tokens [0, sink) ∪ [L - local, L) (oracle), including windows
    that overlap on short requests, an empty sink and an empty local window."""
    w, inp, cache = small(Hq=16, Hkv=4, page=page, L=L, streaming=(1, 3), seed=L + sink)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    G = w.group
    k = 7
    rows = w.batch * 4
    gsel = np.random.default_rng(L)
    idx = np.full((rows, 9), -1, np.int32)
    cnt = np.zeros(rows, np.int32)
    for r in range(rows):
        b, h = divmod(r, 4)
        npos = -(-int(inp["seq_lens"][b]) // page)
        sel = np.sort(gsel.choice(npos, min(k, npos), replace=False))
        idx[r, :len(sel)] = sel
        cnt[r] = len(sel)
    idx_t = torch.tensor(idx, device="cuda").view(w.batch, 4, 9)
    cnt_t = torch.tensor(cnt, device="cuda").view(w.batch, 4)
    out, m, l = cache.outputs()
    ws = torch.zeros(max(16, B.dsa_sparse_decode_attn_workspace_size(cache.kv, 9)),
                     dtype=torch.uint8, device="cuda")
    B.dsa_hybrid_decode_attn(cache.kv, q, idx_t, cnt_t, sink, local, scale, out, m, l, ws)
    torch.cuda.synchronize()
    oc, mc, lc = out.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()
    for b in range(w.batch):
        for h in range(4):
            sl = slice(h * G, (h + 1) * G)
            K, V, Lb = keys_values(inp, cache, b, h)
            if h in (1, 3):
                tok = O.streaming_token_ids(Lb, sink, local)
            else:
                r = b * 4 + h
                tok = O.page_token_ids(idx[r, :cnt[r]], page, Lb)
            ref = O.attend(q[b, sl], K, V, tok, scale)
            assert_outputs(oc[b, sl], mc[b, sl], lc[b, sl], ref, f"hybrid b{b} h{h}")
    assert int(cache.status.item()) == 0


def test_hybrid_matches_two_launches_on_lserve_shape():
    """The LServe workload at oracle scale: one launch equals the dense launch plus the streaming
    launch to fp32 rounding, step after step of the reuse schedule."""
    from dynamic_block_sparse_gb300.pipeline import HierDecoder
    from dynamic_block_sparse_gb300.workloads import BY_NAME, oracle_scale
    w = oracle_scale(BY_NAME["lserve_hier"])
    inp = to_cuda(make_inputs(w, "cpu"))
    outs = []
    for one in (True, False):
        cache = Cache(inp["k_pages"], inp["v_pages"], inp["page_table"], inp["seq_lens"],
                      w.num_q_heads, inp["head_is_streaming"])
        dec = HierDecoder(cache, w.k, w.logical_page, w.sink, w.local, w.reuse, one_launch=one)
        dec.build_meta()
        res = []
        for t in range(w.steps):
            o, m, l = dec.step(inp["q"][t], t)
            res.append([x.double().cpu().numpy() for x in (o, m, l)])
        torch.cuda.synchronize()
        outs.append(res)
    for t in range(w.steps):
        assert_outputs(*outs[0][t], outs[1][t], f"step {t}")


def test_quantize_kv8_matches_oracle_bitwise():
    """KV8 conversion of the whole pool: every code and every row scale equals the oracle's
    encoding (fp32 scale and division, e4m3 rounding to nearest even)."""
    w, inp, cache = small(page=16, L=16 * 30 + 5, seed=41)
    cache.k_pages[3, 1, 5] = 0          # a zero row keeps scale 0
    cache.v_pages[2, 0, :4] *= 1e3      # rows of large magnitude
    buf = cache.kv8()
    torch.cuda.synchronize()
    assert buf.numel() == cache.num_phys_pages * cache.num_kv_heads * 264 * cache.page_size
    k8, v8, ks, vs = B.kv8_unpack(buf, cache.num_phys_pages, cache.num_kv_heads,
                                  cache.page_size)
    for pool, codes, scales in ((cache.k_pages, k8, ks), (cache.v_pages, v8, vs)):
        ref_c, ref_s = O.kv8_encode_rows(pool.float().cpu().numpy())
        np.testing.assert_array_equal(scales.cpu().numpy(), ref_s)
        np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)
    assert float(ks[3, 1, 5]) == 0.0


@pytest.mark.parametrize("page,G", [(16, 4), (64, 16), (32, 1), (16, 8), (32, 2)])
def test_sparse_decode_attn_kv8(page, G):
    """Attention over KV8 pages against the oracle's attention over the decoded rows of the
    selected pages (ragged requests, a short last page); and its distance to the bf16 attention
    stays within the 8-bit format's error.  Groups of at most 8 run the transposed tiles (G = 8 is
    their widest), larger ones the untransposed."""
    Hkv = 2
    w, inp, cache = small(Hq=G * Hkv, Hkv=Hkv, page=page, L=page * 40 + 7, seed=42 + page)
    from dynamic_block_sparse_gb300.pipeline import TopKDecoder
    dec = TopKDecoder(cache, 9)
    dec.build_meta()
    q = inp["q"][0]
    out16, m16, l16 = [x.clone() for x in dec.step(q)]
    dec.use_kv8()
    out, m, l = dec.step(q)
    torch.cuda.synchronize()
    k8, v8, ks, vs = [x.cpu().numpy() for x in B.kv8_unpack(dec.kv8, cache.num_phys_pages,
                                                                cache.num_kv_heads, page)]
    Kd = O.kv8_decode_rows(k8, ks)
    Vd = O.kv8_decode_rows(v8, vs)
    table = cache.page_table.cpu().numpy()
    for b in range(w.batch):
        L = int(cache.seq_lens[b])
        for h in range(Hkv):
            A = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
            toks = O.page_token_ids(A, page, L)
            K = np.stack([Kd[table[b, t // page], h, t % page] for t in range(L)])
            V = np.stack([Vd[table[b, t // page], h, t % page] for t in range(L)])
            sl = slice(h * G, (h + 1) * G)
            ref = O.attend(q[b, sl], K, V, toks, dec.scale)
            assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(),
                           l[b, sl].cpu().numpy(), ref, f"kv8 b{b} h{h}")
    # the 8-bit pages move the output by at most a few percent of its scale
    d = (out - out16).abs().max().item()
    assert d < 0.1 * out16.abs().max().item() + 1e-3
    assert int(cache.status.item()) == 0


def test_quantize_kv4_matches_oracle_bitwise():
    """KV4 conversion of the whole pool: every packed code byte and every row scale equals the
    oracle's encoding (fp32 scale and division, rounding ties to even, offset-8 nibbles)."""
    w, inp, cache = small(page=16, L=16 * 30 + 5, seed=43)
    cache.k_pages[3, 1, 5] = 0          # a zero row keeps scale 0
    cache.v_pages[2, 0, :4] *= 1e3      # rows of large magnitude
    cache.k_pages[1, 0, 2, :8] = torch.tensor([7, -7, 3.5, 0.5, 1.5, 2.5, -2.5, 0],
                                              dtype=torch.bfloat16)  # ties (scale is not 1 here)
    buf = cache.kv4()
    torch.cuda.synchronize()
    assert buf.numel() == cache.num_phys_pages * cache.num_kv_heads * 136 * cache.page_size
    k4, v4, ks, vs = B.kv4_unpack(buf, cache.num_phys_pages, cache.num_kv_heads,
                                  cache.page_size)
    for pool, codes, scales in ((cache.k_pages, k4, ks), (cache.v_pages, v4, vs)):
        ref_c, ref_s = O.kv4_encode_rows(pool.float().cpu().numpy())
        np.testing.assert_array_equal(scales.cpu().numpy(), ref_s)
        np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)
    assert float(ks[3, 1, 5]) == 0.0


@pytest.mark.parametrize("page,G", [(16, 4), (64, 16), (32, 1), (16, 8), (32, 2)])
def test_sparse_decode_attn_kv4(page, G):
    """Attention over KV4 pages against the oracle's attention over the decoded rows of the
    selected pages (ragged requests, a short last page)."""
    Hkv = 2
    w, inp, cache = small(Hq=G * Hkv, Hkv=Hkv, page=page, L=page * 40 + 7, seed=44 + page)
    from dynamic_block_sparse_gb300.pipeline import TopKDecoder
    dec = TopKDecoder(cache, 9)
    dec.build_meta()
    q = inp["q"][0]
    out16 = dec.step(q)[0].clone()
    dec.use_kv4()
    out, m, l = dec.step(q)
    torch.cuda.synchronize()
    k4, v4, ks, vs = [x.cpu().numpy() for x in B.kv4_unpack(dec.kv4, cache.num_phys_pages,
                                                                cache.num_kv_heads, page)]
    Kd = O.kv4_decode_rows(k4, ks)
    Vd = O.kv4_decode_rows(v4, vs)
    table = cache.page_table.cpu().numpy()
    for b in range(w.batch):
        L = int(cache.seq_lens[b])
        for h in range(Hkv):
            A = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
            toks = O.page_token_ids(A, page, L)
            K = np.stack([Kd[table[b, t // page], h, t % page] for t in range(L)])
            V = np.stack([Vd[table[b, t // page], h, t % page] for t in range(L)])
            sl = slice(h * G, (h + 1) * G)
            ref = O.attend(q[b, sl], K, V, toks, dec.scale)
            assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(),
                           l[b, sl].cpu().numpy(), ref, f"kv4 b{b} h{h}")
    # 4-bit pages stay within the format's error of the bf16 attention (half a code step,
    # max|x| / 14 per value, averaged by the softmax)
    d = (out - out16).abs().max().item()
    assert d < 0.5 * out16.abs().max().item() + 1e-2
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("case", ["random", "disjoint", "p_superset", "equal", "empty_p"])
@pytest.mark.parametrize("superset", [False, True])
def test_repair_merge(case, superset):
    w, inp, cache = small(Hq=32, Hkv=2, page=64, L=64 * 50 + 17, seed=11)
    G = w.group
    kA, kP = 10, 12
    g = np.random.default_rng(hash(case) % 997)
    rows = w.batch * 2
    A = np.full((rows, kA), -1, np.int32)
    P = np.full((rows, kP), -1, np.int32)
    cA = np.zeros(rows, np.int32)
    cP = np.zeros(rows, np.int32)
    for r in range(rows):
        b = r // 2
        npos = -(-int(inp["seq_lens"][b]) // 64)
        a = sorted(g.choice(npos, kA, replace=False).tolist())
        rest = [j for j in range(npos) if j not in a]
        if case == "random":
            p = sorted(g.choice(npos, kP, replace=False).tolist())
        elif case == "disjoint":
            p = sorted(g.choice(rest, kP, replace=False).tolist())
        elif case == "p_superset":
            p = sorted(a + g.choice(rest, 2, replace=False).tolist())
        elif case == "equal":
            p = list(a)
        else:
            p = []
        A[r, :len(a)], cA[r] = a, len(a)
        P[r, :len(p)], cP[r] = p, len(p)
    scale = 1 / math.sqrt(128)
    q = inp["q"][0]
    dA, dP = torch.from_numpy(A).cuda(), torch.from_numpy(P).cuda()
    dcA, dcP = torch.from_numpy(cA).cuda(), torch.from_numpy(cP).cuda()
    part = torch.zeros((w.batch, 2, kP, G, B.RECORD_FLOATS), device="cuda")
    B.dsa_sparse_decode_attn(cache.kv, q, dP, dcP, scale, page_partials=part)
    ws = torch.empty(B.dsa_repair_merge_workspace_size(cache.kv, kA), dtype=torch.uint8, device="cuda")
    out, m, l = cache.outputs()
    B.dsa_repair_merge(cache.kv, q, dP, dcP, part, dA, dcA, scale, out, m, l, ws, superset=superset)
    torch.cuda.synchronize()
    for r in range(rows):
        b, h = divmod(r, 2)
        K, V, L = keys_values(inp, cache, b, h)
        sl = slice(h * G, (h + 1) * G)
        pages = sorted(set(A[r, :cA[r]]) | (set(P[r, :cP[r]]) if superset else set()))
        ref = O.attend(q[b, sl], K, V, O.page_token_ids(pages, 64, L), scale)
        orc = O.spec_repair(q[b, sl], K, V, 64, L, P[r, :cP[r]], A[r, :cA[r]], scale, superset)
        for x, y in zip(ref, orc):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)
        assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(), l[b, sl].cpu().numpy(),
                       ref, f"repair {case} row {r}")


# ---------------------------------------------------------------------------------- EMA

def _calib_oracle(traj, rows, n, k, k_pred, points=None):
    """H of the oracle's calibration per row (PRR §3.2), for all grid points or a subset."""
    out = []
    grid = O.calibration_grid()
    for r in range(rows):
        tr = [np.asarray(t[r, :n], dtype=np.float64) for t in traj]
        if points is None:
            _, Hs = O.calibrate_ema(tr, k, k_pred)
            out.append(np.array(Hs))
            continue
        Hs = []
        for c in points:
            a, b, g = grid[c]
            ell, v = O.ema_init(tr[0])
            tot = 0.0
            for t in range(1, len(tr)):
                P = O.select_topk(O.ema_predict(ell, v, g), k_pred)
                A = O.select_topk(tr[t], k)
                tot += O.score_weighted_hit(P, A, tr[t])
                ell, v = O.ema_update(tr[t], ell, v, a, b)
            Hs.append(tot / max(1, len(tr) - 1))
        out.append(np.array(Hs))
    return out


def _calib_gpu(traj, n, k, k_pred, stride):
    steps, rows = len(traj), traj[0].shape[0]
    T = torch.full((steps, rows, stride), -math.inf, device="cuda")
    for t, x in enumerate(traj):
        T[t, :, :n] = x.cuda()
    H = torch.empty((rows, B.CALIB_POINTS), device="cuda")
    best = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.dsa_calibrate_ema_workspace_size(steps, rows, n, k), dtype=torch.uint8,
                     device="cuda")
    B.dsa_calibrate_ema(T, n, k, k_pred, H, best, ws)
    torch.cuda.synchronize()
    assert int(ws[:4 * rows].sum()) == 0, "the row counters are left zero-filled"
    return H.double().cpu().numpy(), best.cpu().numpy()


def test_calibrate_ema_matches_oracle():
    """Every grid point's score-weighted hit rate H against the oracle's calibration (PRR §3.2), on
    drifting trajectories with pages past the request and a page that drops out and comes back;
    the chosen point is the oracle's best up to fp32 selection ties."""
    rows, n, k, k_pred, steps = 3, 700, 24, 29, 9
    gen = torch.Generator().manual_seed(11)
    base = torch.randn(rows, n, generator=gen) * 3 + 100
    slope = torch.randn(rows, n, generator=gen) * 0.8
    traj = [base + slope * t + 0.4 * torch.randn(rows, n, generator=gen) for t in range(steps)]
    for t in traj:
        t[:, n - 60:] = -math.inf                       # pages beyond the request
    traj[4][1, 5:9] = -math.inf                         # a page that drops out, then comes back
    H, best = _calib_gpu(traj, n, k, k_pred, stride=n + 4)
    ref = _calib_oracle(traj, rows, n, k, k_pred)
    for r in range(rows):
        np.testing.assert_allclose(H[r], ref[r], atol=2e-3, rtol=0, err_msg=f"H row {r}")
        assert ref[r][best[r]] >= ref[r].max() - 2e-3, f"row {r}: best {best[r]}"


def test_calibrate_ema_prefers_trend_when_rankings_cross():
    """The crossing-rankings trajectory of the oracle's pins: the GPU also picks a point with
    gamma > 0, and it matches the oracle's choice."""
    n = 40
    slope = np.linspace(-1, 1, n)
    traj = [torch.tensor(np.stack([20 - 6 * slope + slope * t + 0.001 * np.arange(n)] * 2),
                         dtype=torch.float32) for t in range(12)]
    H, best = _calib_gpu(traj, n, 5, 6, stride=48)
    ref = _calib_oracle(traj, 2, n, 5, 6)
    for r in range(2):
        assert B.calibration_point(int(best[r]))[2] > 0
        np.testing.assert_allclose(H[r], ref[r], atol=1e-4, rtol=0)
        assert int(best[r]) == int(np.argmax(ref[r]))


def test_calibrate_ema_full_size_sampled():
    """The PRR 512K shape (2 rows of 8192 blocks, top-64, |P| = 76) over a 16-step random-walk
    trajectory; eight grid points checked against the oracle, and the rest against properties
    (0 <= H <= 1 for positive scores)."""
    rows, n, k, k_pred, steps = 2, 8192, 64, 76, 16
    gen = torch.Generator().manual_seed(12)
    x = torch.randn(rows, n, generator=gen) * 4 + 300
    traj = []
    for _ in range(steps):
        traj.append(x.clone())
        x = x + 0.6 * torch.randn(rows, n, generator=gen)
    H, best = _calib_gpu(traj, n, k, k_pred, stride=n)
    assert np.all((H >= 0) & (H <= 1 + 1e-6))
    points = [0, 7, 22, 39, 41, 58, 63, 79]
    ref = _calib_oracle(traj, rows, n, k, k_pred, points)
    for r in range(rows):
        np.testing.assert_allclose(H[r][points], ref[r], atol=2e-3, rtol=0, err_msg=f"row {r}")
        assert 0 <= best[r] < 80 and H[r][best[r]] == H[r].max()


def test_ema_predict_update_sequence():
    rows, n, k_pred = 3, 5000, 76
    gen = torch.Generator().manual_seed(5)
    base = torch.randn(rows, n, generator=gen) * 3 + 240
    traj = [base + 0.3 * t * torch.randn(rows, n, generator=gen) for t in range(5)]
    for t in traj:
        t[:, n - 100:] = -math.inf                      # pages beyond the request
    traj[3][0, 10:20] = -math.inf                       # temporarily invalid, then fresh again
    stride = n + 8
    IS = torch.full((rows, stride), -math.inf, device="cuda")
    ell = torch.zeros((rows, stride), device="cuda")
    v = torch.zeros_like(ell)
    pred = torch.empty_like(ell)
    pidx = torch.empty((rows, k_pred), dtype=torch.int32, device="cuda")
    pcnt = torch.empty(rows, dtype=torch.int32, device="cuda")
    ell64 = v64 = None
    for t, s in enumerate(traj):
        IS[:, :n] = s.cuda()
        mode = B.DSA_EMA_INIT if t == 0 else B.DSA_EMA_UPDATE
        B.dsa_ema_predict_update(IS, n, ell, v, mode, 0.6, 0.3, 0.5, pred, k_pred, pidx, pcnt)
        torch.cuda.synchronize()
        s64 = s.double().numpy()
        if t == 0:
            ell64, v64 = zip(*[O.ema_init(s64[r]) for r in range(rows)])
        else:
            ell64, v64 = zip(*[O.ema_update(s64[r], ell64[r], v64[r], 0.6, 0.3) for r in range(rows)])
        for r in range(rows):
            lg = ell[r, :n].double().cpu().numpy()
            vg = v[r, :n].double().cpu().numpy()
            fin = np.isfinite(ell64[r])
            assert np.array_equal(np.isneginf(lg), ~fin)
            np.testing.assert_allclose(lg[fin], ell64[r][fin], rtol=1e-6, atol=1e-5)
            np.testing.assert_allclose(vg, v64[r], rtol=1e-5, atol=1e-4)
            p64 = O.ema_predict(ell64[r], v64[r], 0.5)
            check_topk(pidx[r, :pcnt[r]].cpu().numpy(), p64, k_pred, f"P t{t} r{r}")


# ---------------------------------------------------------------------------------- PSA

@pytest.mark.parametrize("tau,cap,nleft,G", [(0.95, 64, False, 1), (0.99, 12, False, 1),
                                             (0.95, 64, True, 1), (1.0, 20, False, 1),
                                             (0.9, 64, False, 4)])
def test_select_threshold(tau, cap, nleft, G):
    w = Workload("psa_unit", 2, 4 * G, 4, 128, 16 * 200 + 3, 16, 16, "mean", "threshold", cap=cap,
                 tau=tau, zipf_s=1.1, seed=21, ragged=True, extra_phys_pages=3)
    inp = to_cuda(make_inputs(w, "cpu"))
    cache = Cache(inp["k_pages"], inp["v_pages"], inp["page_table"], inp["seq_lens"], w.num_q_heads)
    meta = cache.meta_buffer(B.DSA_META_MEAN, 16)
    B.dsa_build_page_meta(cache.kv, B.DSA_META_MEAN, 16, meta)
    stride = cache.max_pages
    scores = torch.empty((w.batch, 4, stride), device="cuda")
    q = inp["q"][0]
    B.dsa_score_pages(cache.kv, q, meta, B.DSA_META_MEAN, 16, scores)
    idx = torch.full((w.batch, 4, cap), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.batch, 4), dtype=torch.int32, device="cuda")
    out, m, l = cache.outputs()
    scale = 1 / math.sqrt(128)
    B.dsa_select_threshold(cache.kv, q, scores, tau, cap, scale, idx, cnt, out, m, l,
                           B.DSA_PSA_NLEFT if nleft else 0)
    torch.cuda.synchronize()
    for b in range(w.batch):
        for h in range(4):
            K, V, L = keys_values(inp, cache, b, h)
            qg = q[b, h * G:(h + 1) * G]
            s64 = oracle_mean_scores(K, qg, 16, stride)
            res = O.psa_progressive(qg, K, V, s64, 16, L, tau, cap, scale, use_nleft=nleft)
            n_gpu = int(cnt[b, h])
            got = idx[b, h, :n_gpu].cpu().numpy().tolist()
            if got != res["ranked"]:
                # allowed only when the decisive ratio sits on the threshold
                r_last = res["ratios"][min(n_gpu, len(res["ratios"])) - 1]
                assert got[:len(res["ranked"])] == res["ranked"][:len(got)], (b, h, got, res["ranked"])
                assert np.min(np.abs(np.asarray(r_last) - tau)) <= 1e-5 * tau, (b, h, n_gpu, len(res["ranked"]))
            ref = O.attend(qg, K, V, O.page_token_ids(got, 16, L), scale)
            sl = slice(h * G, (h + 1) * G)
            assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(), l[b, sl].cpu().numpy(),
                           ref, f"psa b{b} h{h}")


# ---------------------------------------------------------------------------------- robustness

@pytest.mark.parametrize("bad", ["negative", "too_large"])
@pytest.mark.parametrize("path", ["meta", "score", "persistent", "splits", "page_partials",
                                  "streaming", "kv8", "kv4"])
def test_bad_page_id_raises_status_without_fault(bad, path):
    """One bad page-table entry inside a request (negative, or past the pool) per call: the call
    raises DSA_STATUS_BAD_PAGE, skips the page and leaves finite outputs."""
    w, inp, cache = small(Hq=8, Hkv=2, page=16, L=16 * 20, streaming=(1,))
    table = inp["page_table"].clone()
    table[1, 0] = -4 if bad == "negative" else cache.num_phys_pages + 11
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    strm = inp["head_is_streaming"] if path == "streaming" else None
    kv = B.paged_kv(inp["k_pages"], inp["v_pages"], table, inp["seq_lens"], 8, strm, status)
    meta = cache.meta_buffer(B.DSA_META_MINMAX, 16)
    out, m, l = cache.outputs()
    idx = torch.tensor([[[3, 4]] * 2, [[0, 1]] * 2], dtype=torch.int32, device="cuda")
    cnt = torch.full((2, 2), 2, dtype=torch.int32, device="cuda")
    if path != "meta":  # metadata from the intact table (its own status word)
        B.dsa_build_page_meta(cache.kv, B.DSA_META_MINMAX, 16, meta)
    if path == "meta":
        B.dsa_build_page_meta(kv, B.DSA_META_MINMAX, 16, meta)
    elif path == "score":
        scores = torch.empty((2, 2, table.shape[1]), dtype=torch.float32, device="cuda")
        B.dsa_score_pages(kv, inp["q"][0], meta, B.DSA_META_MINMAX, 16, scores)
        torch.cuda.synchronize()
        assert torch.isinf(scores[1, :, 0]).all() and (scores[1, :, 0] < 0).all()
    elif path == "streaming":
        B.dsa_streaming_head_attn(kv, inp["q"][0], 16, 32, 0.1, out, m, l)
    elif path in ("kv8", "kv4"):  # quantised blocks of the whole pool; the bad entry is read
        blocks = cache.kv8() if path == "kv8" else cache.kv4()
        if path == "kv8":
            ws = torch.zeros(max(16, B.dsa_sparse_decode_attn_kv8_workspace_size(kv, 2)),
                             dtype=torch.uint8, device="cuda")
            B.dsa_sparse_decode_attn_kv8(kv, blocks, inp["q"][0], idx, cnt, 0.1, out, m, l, ws)
        else:
            ws = torch.zeros(max(16, B.dsa_sparse_decode_attn_kv4_workspace_size(kv, 2)),
                             dtype=torch.uint8, device="cuda")
            B.dsa_sparse_decode_attn_kv4(kv, blocks, inp["q"][0], idx, cnt, 0.1, out, m, l, ws)
    else:
        splits = {"persistent": 0, "splits": 2, "page_partials": 1}[path]
        parts = None
        if path == "page_partials":
            parts = torch.zeros((2, 2, 2, 4, 132), dtype=torch.float32, device="cuda")
        ws = torch.zeros(max(16, B.dsa_sparse_decode_attn_workspace_size(kv, 2, splits)),
                         dtype=torch.uint8, device="cuda")
        B.dsa_sparse_decode_attn(kv, inp["q"][0], idx, cnt, 0.1, out, m, l,
                                 page_partials=parts, num_splits=splits, workspace=ws)
        if parts is not None:
            torch.cuda.synchronize()
            assert torch.isfinite(parts[..., :128]).all() and torch.isfinite(parts[..., 129]).all()
    torch.cuda.synchronize()
    assert int(status.item()) == B.DSA_STATUS_BAD_PAGE
    assert torch.isfinite(out).all() and torch.isfinite(l).all()


def test_host_errors_are_reported():
    w, inp, cache = small()
    kv = B.paged_kv(inp["k_pages"], inp["v_pages"], inp["page_table"], inp["seq_lens"], 8)
    kv.head_dim = 64
    with pytest.raises(B.DsaError, match="head_dim"):
        B.dsa_build_page_meta(kv, 0, 16, cache.meta_buffer(0, 16))
    scores = torch.zeros((2, 10), device="cuda")
    with pytest.raises(B.DsaError, match="idx_stride"):
        B.dsa_select_topk(scores, 10, 5, torch.zeros((2, 3), dtype=torch.int32, device="cuda"),
                          torch.zeros(2, dtype=torch.int32, device="cuda"))


def test_kernels_are_deterministic():
    w, inp, cache = small(Hq=32, Hkv=2, page=64, L=64 * 60, seed=1)
    idx, cnt = _random_selection(w, inp, 40, seed=2, allow_bad=False)
    dI, dC = torch.from_numpy(idx).cuda(), torch.from_numpy(cnt).cuda()
    ws = torch.zeros(B.dsa_sparse_decode_attn_workspace_size(cache.kv, 40) + 16,
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out, m, l = cache.outputs()
        B.dsa_sparse_decode_attn(cache.kv, inp["q"][0], dI, dC, 0.08, out, m, l, workspace=ws)
        outs.append((out.clone(), m.clone(), l.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
