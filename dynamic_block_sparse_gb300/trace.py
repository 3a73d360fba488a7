"""Phase timelines of the fused kernels, read from the tracing build of the library.

    python -m dynamic_block_sparse_gb300.trace threshold   # PSA threshold kernel on psa_threshold
    python -m dynamic_block_sparse_gb300.trace prr         # fused PRR step on prr_512k
    python -m dynamic_block_sparse_gb300.trace stream      # persistent attention on llama3_8b_layer
    python -m dynamic_block_sparse_gb300.trace stream --pages kv8   # the same over KV8 (or kv4) pages

Builds ``libdsa_trace.so`` (every kernel compiled with ``-DDSA_TIMELINE``), runs the workload's
step several times cold (L2 flushed before each launch) and warm (launches back to back), and
prints for every stamp the median and the maximum over the CTAs of all runs: clock64 cycles since
the CTA's own start, and %globaltimer nanoseconds since the earliest CTA start of the launch.  The
tracing build adds a barrier at each instrumented kernel's start and a few tens of cycles per
stamp; the stamps bound phases approximately (the compiler orders them against the surrounding
code only as it orders volatile operations).  The fused PRR step's CTAs are reported by role:
workers (scoring, speculative pages), merge task CTAs (A_t, repair, merge) and the P_{t+1}
selection CTAs.
"""

from __future__ import annotations

import argparse
import ctypes
import statistics
import sys

import numpy as np

LABELS = {
    "threshold": {
        1: "score row landed",
        2: "keys converted, two largest per thread",
        3: "warp keys shared (barrier)",
        4: "chunk bound",
        5: "candidates collected (barrier)",
        6: "ranked (barrier)",
        7: "page-table entries done, TMA issued",
        8: "pages landed",
        9: "block masses (barrier)",
        10: "stop rule decided",
        11: "P.V done (thread 0's warp)",
        12: "chunk done (barrier)",
        13: "warp states merged, output written",
    },
    "stream": {
        1: "set-up done (barrier)",
        2: "first unit's descriptor and query on chip (consumer warp 0)",
        3: "warp 0's first page landed",
        4: "warp 0 through the first unit's pages",
        5: "the first unit's epilogue done",
        6: "the consumers' work done (end)",
        8: "producer: its first page loads issued",
        9: "producer: every load issued",
        10: "producer: first batch's unit descriptors known",
        11: "producer: the first unit published (mailbox, query copy)",
        12: "producer: first chunk about to issue (page-table entries in hand)",
        13: "producer: partition known",
        14: "last unit: every warp's state stored (its pages done)",
        15: "last unit: epilogue done",
        16: "cut rows: tickets taken",
        17: "cut rows: merge done (merging CTAs)",
        18: "producer: the general loop's first loads issued",
        19: "producer: set-up done (arrived)",
        20: "last unit: thread 0's share of the epilogue done",
        21: "cut rows: thread 0's ticket returned",
        22: "warp 0: its fourth page landed",
        23: "warp 0: its fourth page attended and released",
        24: "warp 0: waiting for its fourth page",
    },
    "prr": {
        1: "worker: first segment's table, state and query loaded",
        2: "worker: share scored, EMA updated, published",
        3: "worker: compute warps' part over (thread 0)",
        4: "worker part and this CTA's P_t pages over (barrier)",
        5: "task: start",
        6: "task: the row's scores complete",
        7: "task: A_t candidates (next-P: the keys) loaded",
        8: "task: ranked, records fetched (barrier)",
        9: "task: merged and missed lists",
        10: "task: missed pages attended",
        11: "task: records ready",
        12: "task: output written",
        13: "end",
        14: "task: A_t ranked from the candidate list (compute warps)",
        15: "task: A_t from the row's keys (no usable list)",
        16: "worker: first round's record loads issued",
        17: "worker: thread 0's first-round scores and EMA written",
        18: "worker: first segment's rounds done (barrier)",
        19: "task: thread 0's warp has merged its records",
        20: "task: every warp's merge state stored (barrier)",
    },
}
SLOTS = 32
CTAS = 1024


def _flusher(torch, dev):
    wbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(64 << 20, dtype=torch.int32, device=dev)
    sink = torch.empty((), dtype=torch.int32, device=dev)

    def flush(i):
        wbuf.fill_(i & 255)
        torch.amax(rbuf, dim=0, out=sink)
    return flush


def _setup(kernel, B, torch, pages="bf16"):
    from dynamic_block_sparse_gb300.pipeline import Cache, PRRDecoder, ThresholdDecoder
    from dynamic_block_sparse_gb300.workloads import BY_NAME, make_inputs

    if kernel == "stream":
        from dynamic_block_sparse_gb300.pipeline import TopKDecoder
        w = BY_NAME["llama3_8b_layer"]
        inp = make_inputs(w, "cuda", shuffle_pages=False)
        cache = Cache.from_inputs(inp, "cuda")
        dec = TopKDecoder(cache, w.k, w.logical_page)
        dec.build_meta()
        q = inp["q"][0].clone()
        dec.step(q)
        if pages == "kv8":
            dec.use_kv8()
        elif pages == "kv4":
            dec.use_kv4()

        def step(i):
            dec.attend(q)
        return step, cache
    if kernel == "threshold":
        w = BY_NAME["psa_threshold"]
        inp = make_inputs(w, "cuda", shuffle_pages=False)
        cache = Cache.from_inputs(inp, "cuda")
        dec = ThresholdDecoder(cache, w.tau, w.cap)
        dec.build_meta()
        q = inp["q"][0].clone()
        dec.step(q)

        def step(i):
            B.dsa_select_threshold(cache.kv, q, dec.scores, w.tau, w.cap, dec.scale, dec.idx,
                                   dec.count, dec.out, dec.m, dec.l)
        return step, cache
    w = BY_NAME["prr_512k"]
    inp = make_inputs(w, "cuda", shuffle_pages=False)
    cache = Cache.from_inputs(inp, "cuda")
    dec = PRRDecoder(cache, w.k, w.k_pred, w.alpha, w.beta, w.gamma)
    dec.build_meta()
    qs = inp["q"]
    q = qs[0].clone()
    dec.step(q)
    for i in range(1, 4):
        q.copy_(qs[i])
        dec.step(q)

    def step(i):
        q.copy_(qs[4 + i % (qs.shape[0] - 4)])
        dec.step(q)
    return step, cache


def _collect(kernel, lib, step, flush, torch, cold: bool, runs: int):
    read = getattr(lib, f"dsa_trace_read_{kernel}")
    clear = getattr(lib, f"dsa_trace_clear_{kernel}")
    read.argtypes, read.restype = [ctypes.c_void_p, ctypes.c_size_t], ctypes.c_int
    clear.argtypes, clear.restype = [], ctypes.c_int
    out = []
    for i in range(runs):
        if clear() != 0:
            raise RuntimeError("trace clear failed")
        torch.cuda.synchronize()
        if cold:
            flush(i)
        else:
            step(i)  # the launch before the traced one: code and data warm
        if not cold:
            if clear() != 0:
                raise RuntimeError("trace clear failed")
        step(i)
        torch.cuda.synchronize()
        buf = np.zeros(CTAS * 2 * SLOTS, dtype=np.uint64)
        if read(buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes) != 0:
            raise RuntimeError("trace read failed")
        out.append(buf.reshape(CTAS, 2, SLOTS).astype(np.int64))
    return out


# phase lengths worth reading per CTA (stamp pairs, both passed by the same CTA)
SPANS = {
    "prr": [(5, 6), (6, 7), (7, 14), (14, 8), (8, 9), (9, 10), (10, 11), (11, 19), (19, 20),
            (20, 12), (12, 13)],
    "stream": [(0, 19), (19, 13), (13, 12), (12, 8), (8, 3), (8, 18), (1, 2), (3, 4), (4, 5),
               (14, 20), (20, 15), (15, 21), (21, 16), (16, 17), (16, 6), (9, 6), (24, 22),
               (22, 23)],
}


def _spans(kernel, runs):
    pairs = SPANS.get(kernel)
    if not pairs:
        return
    print("   per-CTA phase lengths (cycles; median / max over the CTAs that passed both stamps)")
    for a, b in pairs:
        d = []
        for tr in runs:
            hit = (tr[:, 0, a] > 0) & (tr[:, 0, b] > 0)
            if a == 0:
                hit &= tr[:, 0, 0] > 0
            d += (tr[hit, 0, b] - tr[hit, 0, a]).tolist()
        if d:
            print(f"   {a:2d} -> {b:2d}  median {int(statistics.median(d)):7d}  max {max(d):7d}"
                  f"   ({len(d)} CTA spans)")


def _report(kernel, runs, title):
    labels = LABELS[kernel]
    groups = {"all CTAs": None}
    if kernel == "prr":  # by the first stamp only that role passes (next-P: 6 without 5)
        groups = {"worker CTAs": 1, "merge task CTAs": 5, "next-P selection CTAs": -6}
    print(f"-- {title}")
    for gname, marker in groups.items():
        cyc = {k: [] for k in labels}
        ns = {k: [] for k in labels}
        n_ctas = 0
        for tr in runs:
            started = tr[:, 0, 0] > 0
            if not started.any():
                continue
            g0 = tr[started, 1, 0].min()
            if marker is None:
                sel = started
            elif marker > 0:
                sel = started & (tr[:, 0, marker] > 0)
            else:
                sel = started & (tr[:, 0, -marker] > 0) & (tr[:, 0, 5] == 0)
            n_ctas += int(sel.sum())
            for k in labels:
                hit = sel & (tr[:, 0, k] > 0)
                cyc[k] += (tr[hit, 0, k] - tr[hit, 0, 0]).tolist()
                ns[k] += (tr[hit, 1, k] - g0).tolist()
        print(f"   {gname} ({n_ctas // max(1, len(runs))} per launch)"
              f"{'':14s} cycles since CTA start        ns since launch start")
        for k, name in labels.items():
            if not cyc[k]:
                continue
            print(f"   {k:2d} {name:46s} median {int(statistics.median(cyc[k])):7d} max "
                  f"{max(cyc[k]):7d}   median {int(statistics.median(ns[k])):7d} max {max(ns[k]):7d}"
                  f"   ({len(cyc[k])} CTA stamps)")
    _spans(kernel, runs)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("kernel", choices=sorted(LABELS))
    p.add_argument("--runs", type=int, default=5)
    p.add_argument("--pages", choices=["bf16", "kv8", "kv4"], default="bf16",
                   help="page format of the stream trace")
    args = p.parse_args(argv)
    import torch

    from dynamic_block_sparse_gb300 import binding as B
    from dynamic_block_sparse_gb300 import build as Bd

    if not torch.cuda.is_available():
        raise SystemExit("the tracing build runs on a CUDA device")
    lib = B.load(Bd.build_traced())
    step, cache = _setup(args.kernel, B, torch, args.pages)
    flush = _flusher(torch, "cuda")
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    _report(args.kernel, _collect(args.kernel, lib, step, flush, torch, True, args.runs),
            f"{args.kernel}: cold launches (L2 flushed before each), {args.runs} runs")
    _report(args.kernel, _collect(args.kernel, lib, step, flush, torch, False, args.runs),
            f"{args.kernel}: warm launches (right after the same step), {args.runs} runs")
    if int(cache.status.item()) != 0:
        raise SystemExit(f"device status raised: {int(cache.status.item())}")


if __name__ == "__main__":
    sys.exit(main())
