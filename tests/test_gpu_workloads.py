"""End-to-end parity of the five decode workloads against the float64 oracle.

Each workload runs through its pipeline (the library calls in production order).  At oracle scale
every row of every step is checked; at full size (the shapes and launch configuration the bench
times) a sample of rows is checked against the oracle computed row by row.
"""

import math
import time

import numpy as np
import pytest
import torch

import oracle as O
from dynamic_block_sparse_gb300 import binding as B
from dynamic_block_sparse_gb300.pipeline import (Cache, HierDecoder, PRRDecoder, ThresholdDecoder,
                                                 TopKDecoder)
from dynamic_block_sparse_gb300.workloads import BY_NAME, WORKLOADS, make_inputs, oracle_scale
from support import (assert_close, assert_outputs, attend_pages, check_ranking, check_topk,
                     row_meta_minmax, row_tokens, to_cuda)

pytestmark = pytest.mark.gpu


def _rows(w, sample):
    rows = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    if sample is None:
        return rows
    g = np.random.default_rng(w.seed)
    pick = sorted(g.choice(len(rows), min(sample, len(rows)), replace=False).tolist())
    return [rows[i] for i in pick]


_META_CACHE = {}   # oracle kmax/kmin per row of the workload being run; cleared per run


def _minmax_scores(inp, b, h, lp, stride, q_group):
    """Oracle page scores of one row; the row's kmax/kmin (fixed across decode steps) is computed
    once per input set."""
    L = int(inp["seq_lens"][b])
    key = (b, h, lp)
    if key not in _META_CACHE:
        _META_CACHE[key] = row_meta_minmax(inp["k_pages"], inp["page_table"], L, b, h, lp)
    kmax, kmin = _META_CACHE[key]
    s = O.score_pages_minmax(O.representative_query(q_group), kmax, kmin)
    return O.pad_scores(s, stride)


def run_topk(w, inp, sample):
    _META_CACHE.clear()
    cache = Cache.from_inputs(inp)
    dec = TopKDecoder(cache, w.k, w.logical_page)
    dec.build_meta()
    q = inp["q"][0]
    out, m, l = dec.step(q)
    torch.cuda.synchronize()
    G = w.group
    exact = 0
    for b, h in _rows(w, sample):
        L = int(inp["seq_lens"][b])
        qg = q[b, h * G:(h + 1) * G]
        s64 = _minmax_scores(inp, b, h, w.logical_page, dec.stride, qg)
        gs = dec.scores[b, h].double().cpu().numpy()
        nl = -(-L // w.logical_page)
        assert_close(gs[:nl], s64[:nl], f"scores b{b} h{h}")
        sel = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
        exact += check_topk(sel, s64, w.k, f"topk b{b} h{h}")
        ref = attend_pages(qg, inp["k_pages"], inp["v_pages"], inp["page_table"], L, b, h, sel,
                           w.scale)
        sl = slice(h * G, (h + 1) * G)
        assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(), l[b, sl].cpu().numpy(),
                       ref, f"out b{b} h{h}")
    assert int(cache.status.item()) == 0
    return exact


def run_hier(w, inp, sample):
    _META_CACHE.clear()
    cache = Cache.from_inputs(inp)
    dec = HierDecoder(cache, w.k, w.logical_page, w.sink, w.local, w.reuse)
    dec.build_meta()
    G = w.group
    rows = _rows(w, sample)
    sel_at = {}
    for t in range(w.steps):
        q = inp["q"][t]
        out, m, l = dec.step(q, t)
        torch.cuda.synchronize()
        for b, h in rows:
            L = int(inp["seq_lens"][b])
            qg = q[b, h * G:(h + 1) * G]
            sl = slice(h * G, (h + 1) * G)
            if h in w.streaming_kv_heads:
                K = row_tokens(inp["k_pages"], inp["page_table"], L, b, h)
                V = row_tokens(inp["v_pages"], inp["page_table"], L, b, h)
                ref = O.attend(qg, K, V, O.streaming_token_ids(L, w.sink, w.local), w.scale)
            else:
                if t % w.reuse == 0:
                    s64 = _minmax_scores(inp, b, h, w.logical_page, dec.stride, qg)
                    phys = O.physical_scores(s64, w.g)
                    sel = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
                    check_topk(sel, phys, w.k, f"hier t{t} b{b} h{h}")
                    sel_at[(b, h)] = sel
                ref = attend_pages(qg, inp["k_pages"], inp["v_pages"], inp["page_table"], L, b, h,
                                   sel_at[(b, h)], w.scale)
            assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(),
                           l[b, sl].cpu().numpy(), ref, f"t{t} b{b} h{h}")
    assert int(cache.status.item()) == 0


def run_threshold(w, inp, sample):
    _META_CACHE.clear()
    cache = Cache.from_inputs(inp)
    dec = ThresholdDecoder(cache, w.tau, w.cap)
    dec.build_meta()
    q = inp["q"][0]
    out, m, l = dec.step(q)
    torch.cuda.synchronize()
    G = w.group
    counts = []
    for b, h in _rows(w, sample):
        L = int(inp["seq_lens"][b])
        qg = q[b, h * G:(h + 1) * G]
        K = row_tokens(inp["k_pages"], inp["page_table"], L, b, h)
        V = row_tokens(inp["v_pages"], inp["page_table"], L, b, h)
        s64 = O.pad_scores(O.score_pages_mean(O.representative_query(qg), O.page_meta_mean(K, w.page_size)),
                           dec.stride)
        res = O.psa_progressive(qg, K, V, s64, w.page_size, L, w.tau, w.cap, w.scale)
        n = int(dec.count[b, h])
        got = dec.idx[b, h, :n].cpu().numpy().tolist()
        check_ranking(got, s64, f"psa b{b} h{h}")
        if n != len(res["ranked"]):
            k = min(n, len(res["ranked"]))
            r_dec = np.asarray(res["ratios"][k - 1])
            assert np.min(np.abs(r_dec - w.tau)) <= 1e-5 * w.tau, (b, h, n, len(res["ranked"]))
        counts.append(n)
        ref = O.attend(qg, K, V, O.page_token_ids(got, w.page_size, L), w.scale)
        sl = slice(h * G, (h + 1) * G)
        assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(), l[b, sl].cpu().numpy(),
                       ref, f"psa out b{b} h{h}")
        if got == res["ranked"]:
            assert_close(out[b, sl].cpu().numpy(), res["O_fused"], f"psa fused b{b} h{h}")
    assert int(cache.status.item()) == 0
    return counts


def run_prr(w, inp, sample, superset=False, fused=True):
    _META_CACHE.clear()
    cache = Cache.from_inputs(inp)
    dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma, superset=superset,
                     fused=fused)
    dec.build_meta()
    G = w.group
    rows = _rows(w, sample)
    state = {}
    hits = []
    for t in range(w.steps):
        q = inp["q"][t]
        P_gpu = dec.spec_idx.clone()
        P_cnt = dec.spec_count.clone()
        out, m, l = dec.step(q)
        torch.cuda.synchronize()
        for b, h in rows:
            L = int(inp["seq_lens"][b])
            qg = q[b, h * G:(h + 1) * G]
            IS = _minmax_scores(inp, b, h, w.page_size, dec.stride, qg)
            A = dec.idx[b, h, :int(dec.count[b, h])].cpu().numpy()
            check_topk(A, IS, w.k, f"A t{t} b{b} h{h}")
            pages = set(A.tolist())
            if t == 0:
                state[(b, h)] = O.ema_init(IS)
            else:
                ell, v = state[(b, h)]
                pred = O.ema_predict(ell, v, w.gamma)
                P = P_gpu[b, h, :int(P_cnt[b, h])].cpu().numpy()
                check_topk(P, pred, w.k_pred, f"P t{t} b{b} h{h}")
                hits.append(O.hit_rate(P, A))
                if superset:
                    pages |= set(P.tolist())
                state[(b, h)] = O.ema_update(IS, ell, v, w.alpha, w.beta)
            ref = attend_pages(qg, inp["k_pages"], inp["v_pages"], inp["page_table"], L, b, h,
                               sorted(pages), w.scale)
            sl = slice(h * G, (h + 1) * G)
            assert_outputs(out[b, sl].cpu().numpy(), m[b, sl].cpu().numpy(),
                           l[b, sl].cpu().numpy(), ref, f"prr t{t} b{b} h{h}")
            # the EMA state on the GPU tracks the oracle's
            ell64, v64 = state[(b, h)]
            fin = np.isfinite(ell64)
            assert_close(dec.ell[b, h].double().cpu().numpy()[fin], ell64[fin], f"ell t{t}")
    assert int(cache.status.item()) == 0
    return hits


RUNNERS = {"topk": run_topk, "hier": run_hier, "threshold": run_threshold, "prr": run_prr}


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_workload_at_oracle_scale(name):
    w = oracle_scale(BY_NAME[name])
    inp = to_cuda(make_inputs(w, "cpu"))
    RUNNERS[w.mode](w, inp, None)


def test_prr_superset_mode_at_oracle_scale():
    w = oracle_scale(BY_NAME["prr_512k"])
    inp = to_cuda(make_inputs(w, "cpu"))
    run_prr(w, inp, None, superset=True)


@pytest.mark.parametrize("superset", [False, True])
def test_prr_staged_path_at_oracle_scale(superset):
    """The separate-launch path (three streams) against the oracle, as the fused path above."""
    w = oracle_scale(BY_NAME["prr_512k"])
    inp = to_cuda(make_inputs(w, "cpu"))
    run_prr(w, inp, None, superset=superset, fused=False)


def _prr_fused_vs_staged(w, inp, superset):
    """Runs the fused one-launch step and the separate-launch step side by side: scores, both
    selections, the EMA state and the prediction agree bit for bit; the partial records and the
    outputs agree to fp32 rounding."""
    decs = []
    for fused in (True, False):
        cache = Cache.from_inputs(inp)
        dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma, superset=superset,
                         fused=fused)
        dec.build_meta()
        decs.append(dec)
    for t in range(w.steps):
        for dec in decs:
            dec.step(inp["q"][t])
        torch.cuda.synchronize()
        f, s = decs
        for name in ("scores", "ell", "trend", "pred", "idx", "count"):
            assert torch.equal(getattr(f, name), getattr(s, name)), f"{name} differs at step {t}"
        assert torch.equal(f.spec_idx, s.spec_idx) and torch.equal(f.spec_count, s.spec_count)
        if t > 0:
            P_cnt = s.spec_counts[(t - 1) % 2]
            for r in range(P_cnt.numel()):
                b, h = divmod(r, w.num_kv_heads)
                n = int(P_cnt[b, h])
                rec_f = f.partials[b, h, :n].double().cpu().numpy()
                rec_s = s.partials[b, h, :n].double().cpu().numpy()
                assert_close(rec_f[..., :130], rec_s[..., :130], f"records t{t} b{b} h{h}")
        assert_outputs(f.out.cpu().numpy(), f.m.cpu().numpy(), f.l.cpu().numpy(),
                       [x.double().cpu().numpy() for x in (s.out, s.m, s.l)], f"step {t}")
        assert int(f.cache.status.item()) == 0
    ws = decs[0].step_workspace
    nctr = B.dsa_prr_step_counter_bytes(decs[0].cache.kv)
    assert nctr > 0 and int(ws[:nctr].sum()) == 0, "the step's counters were not left at zero"


@pytest.mark.parametrize("superset", [False, True])
def test_prr_fused_step_matches_staged_at_oracle_scale(superset):
    w = oracle_scale(BY_NAME["prr_512k"])
    _prr_fused_vs_staged(w, to_cuda(make_inputs(w, "cpu")), superset)


# Shapes that take the fused step's other paths: more rows than half the CTAs (every CTA selects,
# waits, then updates the EMA and repairs), a small group on 16-token pages (one tile per page,
# G = 4), and ragged requests with pages past the end of the shorter ones.
@pytest.mark.parametrize("shape", ["many_rows", "g4_page16", "ragged", "wide_table"])
def test_prr_fused_step_shapes(shape):
    base = BY_NAME["prr_512k"]
    if shape == "wide_table":
        # a page table far wider than the requests: each CTA's share of the score rows is too big
        # to stage the EMA update on chip, so the update runs after scoring instead
        w = base.replace(batch=4, seq_len=64 * 100 + 9, k=12, steps=4, ragged=True)
        inp = to_cuda(make_inputs(w, "cpu"))
        table = inp["page_table"]
        inp["page_table"] = torch.cat(
            [table, torch.zeros((table.shape[0], 20000 - table.shape[1]), dtype=table.dtype,
                                device=table.device)], dim=1).contiguous()
        _prr_fused_vs_staged(w, inp, False)
        return
    if shape == "many_rows":
        w = base.replace(batch=48, num_kv_heads=2, num_q_heads=32, seq_len=64 * 40 + 7, k=8,
                         steps=3, ragged=True, extra_phys_pages=3)
    elif shape == "g4_page16":
        w = base.replace(batch=3, num_q_heads=8, num_kv_heads=2, seq_len=16 * 300 + 5,
                         page_size=16, logical_page=16, k=20, steps=4, ragged=True)
    else:
        w = base.replace(batch=5, seq_len=64 * 90, k=12, steps=4, ragged=True,
                         extra_phys_pages=9)
    _prr_fused_vs_staged(w, to_cuda(make_inputs(w, "cpu")), shape == "ragged")


def test_prr_fused_step_matches_staged_full_size():
    w = BY_NAME["prr_512k"].replace(steps=6)
    _prr_fused_vs_staged(w, make_inputs(w, "cuda"), False)


def test_prr_without_second_stream_matches():
    w = oracle_scale(BY_NAME["prr_512k"]).replace(steps=3)
    inp = to_cuda(make_inputs(w, "cpu"))
    outs = []
    for two in (True, False):
        cache = Cache.from_inputs(inp)
        dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma, two_streams=two,
                         fused=False)
        dec.build_meta()
        for t in range(w.steps):
            dec.step(inp["q"][t])
        torch.cuda.synchronize()
        outs.append(dec.out.clone())
    assert torch.equal(outs[0], outs[1])


def test_prr_decoder_calibrates_on_its_score_trajectory():
    """PRRDecoder.calibrate rates the grid on a trajectory of the workload's own true scores (the
    scoring call over a random-walking query) and adopts the majority point; the rates match the
    oracle's calibration on sampled grid points."""
    w = oracle_scale(BY_NAME["prr_512k"]).replace(steps=8)
    inp = to_cuda(make_inputs(w, "cpu"))
    dec = PRRDecoder(Cache.from_inputs(inp), w.k, w.k_pred, w.alpha, w.beta, w.gamma)
    dec.build_meta()
    traj = torch.empty((w.steps,) + tuple(dec.scores.shape), device="cuda")
    for t in range(w.steps):
        dec.stage_score(inp["q"][t])
        traj[t].copy_(dec.scores)
    H, best = dec.calibrate(traj)
    torch.cuda.synchronize()
    rows = traj.shape[1] * traj.shape[2]
    t3 = traj.view(w.steps, rows, -1).cpu().double().numpy()
    grid = O.calibration_grid()
    for r in range(rows):
        n = int(np.isfinite(t3[0, r]).sum())
        tr = [t3[t, r, :n] for t in range(w.steps)]
        for c in (0, 13, 42, int(best[r])):
            a, b, g = grid[c]
            ell, v = O.ema_init(tr[0])
            tot = 0.0
            for t in range(1, w.steps):
                P = O.select_topk(O.ema_predict(ell, v, g), w.k_pred)
                A = O.select_topk(tr[t], w.k)
                tot += O.score_weighted_hit(P, A, tr[t])
                ell, v = O.ema_update(tr[t], ell, v, a, b)
            assert abs(float(H[r, c]) - tot / (w.steps - 1)) < 2e-3, f"row {r} point {c}"
    assert (dec.alpha, dec.beta, dec.gamma) == B.calibration_point(
        int(torch.bincount(best.long(), minlength=80).argmax()))


def test_prr_decode_loop_with_kv_append():
    """PRR decoding while the context grows: before every step each request appends a token
    (metadata kept by the append, never rebuilt), opening new pages along the way.  The fused step
    and the separate-launch path agree bit for bit on scores, selections and the EMA state (new
    pages start fresh), and to fp32 rounding on the outputs."""
    w = oracle_scale(BY_NAME["prr_512k"]).replace(steps=10, ragged=True, batch=2)
    inp = to_cuda(make_inputs(w, "cpu"))
    grow = 2 * w.page_size + 5
    decs = []
    for fused in (True, False):
        # each decoder grows its own copy of the cache (inputs already on the device are not
        # copied by Cache.from_inputs)
        own = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in inp.items()}
        cache = Cache.from_inputs(own)
        cache.seq_lens.sub_(grow)
        dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma, fused=fused)
        dec.build_meta()
        decs.append(dec)
    f, s_ = decs
    gen = torch.Generator(device="cuda").manual_seed(31)
    shape = (w.batch, w.num_kv_heads, 128)
    for t in range(w.steps):
        for _ in range(grow // w.steps):
            k_new = torch.randn(shape, generator=gen, device="cuda").bfloat16()
            v_new = torch.randn(shape, generator=gen, device="cuda").bfloat16()
            for dec in decs:
                dec.append(k_new, v_new)
        for dec in decs:
            dec.step(inp["q"][t % inp["q"].shape[0]])
        torch.cuda.synchronize()
        assert torch.equal(f.cache.k_pages, s_.cache.k_pages)
        assert torch.equal(f.meta, s_.meta)
        for name in ("scores", "ell", "trend", "idx", "count"):
            assert torch.equal(getattr(f, name), getattr(s_, name)), f"{name} at step {t}"
        assert_outputs(f.out.cpu().numpy(), f.m.cpu().numpy(), f.l.cpu().numpy(),
                       [x.double().cpu().numpy() for x in (s_.out, s_.m, s_.l)], f"step {t}")
        assert int(f.cache.status.item()) == 0 and int(s_.cache.status.item()) == 0


def test_prr_step_with_host_query_and_result():
    """The fused step with its query and its result (O, m, l) in page-locked host memory, which the
    kernel reads and writes over the host link itself, gives the same scores, selections, EMA
    state and outputs as with device buffers."""
    w = oracle_scale(BY_NAME["prr_512k"]).replace(steps=5)
    inp = to_cuda(make_inputs(w, "cpu"))
    decs = []
    for _ in range(2):
        dec = PRRDecoder(Cache.from_inputs(inp), w.k, w.k_pred, w.alpha, w.beta, w.gamma)
        dec.build_meta()
        dec.step(inp["q"][0])  # step 0 (separate launches) takes device buffers only
        decs.append(dec)
    dev, host = decs
    host.host_result()
    assert not host.out.is_cuda and host.out.is_pinned()
    q_host = inp["q"].cpu().pin_memory()
    for t in range(1, w.steps):
        dev.step(inp["q"][t])
        host.step(q_host[t])
        torch.cuda.synchronize()
        for name in ("scores", "ell", "trend", "pred", "idx", "count"):
            assert torch.equal(getattr(dev, name), getattr(host, name)), f"{name} at step {t}"
        assert_outputs(host.out.numpy(), host.m.numpy(), host.l.numpy(),
                       [x.double().cpu().numpy() for x in (dev.out, dev.m, dev.l)], f"step {t}")
        assert int(host.cache.status.item()) == 0


def test_prr_step_wait_timeout_sets_status():
    """Failure detection without a fault: every per-row counter of the fused step starts at
    -2^30, so the increments of all CTAs still leave each one short of its target (a flag that
    nothing sets; the waits compare counters as sequence numbers).  Each bounded wait gives up after its limit, the kernel returns early with
    DSA_STATUS_TIMEOUT in the status word, and the context stays usable: with the counters and
    the status zeroed again, the next step selects A_t exactly as the staged path does and attends
    over it."""
    w = BY_NAME["prr_512k"].replace(seq_len=65536, steps=4)
    inp = make_inputs(w, "cuda")
    decs = []
    for fused in (True, False):
        cache = Cache.from_inputs(inp)
        dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma, fused=fused)
        dec.build_meta()
        decs.append(dec)
    f, s = decs
    for t in range(2):
        for dec in decs:
            dec.step(inp["q"][t])
    torch.cuda.synchronize()
    ws = f.step_workspace
    nctr = B.dsa_prr_step_counter_bytes(f.cache.kv)
    ws[:nctr].view(torch.int32).fill_(-(1 << 30))
    t0 = time.monotonic()
    f.step(inp["q"][2])
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(f.cache.status.item()) & B.DSA_STATUS_TIMEOUT, "the unreachable barrier went unseen"
    assert elapsed < 60.0, f"the bounded waits took {elapsed:.1f} s"
    s.step(inp["q"][2])
    # recovery: the caller zeroes the workspace and the status, then steps on
    ws.zero_()
    f.cache.status.zero_()
    for dec in decs:
        dec.step(inp["q"][3])
    torch.cuda.synchronize()
    assert int(f.cache.status.item()) == 0
    assert torch.equal(f.scores, s.scores)
    assert torch.equal(f.idx, s.idx) and torch.equal(f.count, s.count)
    assert_outputs(f.out.cpu().numpy(), f.m.cpu().numpy(), f.l.cpu().numpy(),
                   [x.double().cpu().numpy() for x in (s.out, s.m, s.l)], "step after recovery")


SAMPLE = {"tiny_topk": None, "llama3_8b_layer": 4, "lserve_hier": 3, "psa_threshold": 4,
          "prr_512k": None}


@pytest.mark.slow
@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_workload_full_size(name):
    w = BY_NAME[name]
    inp = make_inputs(w, "cuda")
    res = RUNNERS[w.mode](w, inp, SAMPLE[name])
    if name == "prr_512k":
        assert np.mean(res) > 0.5        # diagnostic floor: the predictor is far better than chance
    _META_CACHE.clear()
    del inp
    torch.cuda.empty_cache()
