"""Decode-step pipelines over libdsa: host-side sequencing of the C-ABI calls, nothing else.

Every buffer a step needs is allocated once, when a decoder is built; a step only enqueues
library kernels on the current CUDA stream (and, for PRR, on a second stream).

* :class:`TopKDecoder`      — kmax/kmin page scores, fixed top-K, sparse attention.
* :class:`HierDecoder`      — LServe: logical pages scored, max-reduced to physical pages,
                              top-K physical pages reused for ``reuse`` steps; streaming heads
                              attend to their sink + local window.
* :class:`ThresholdDecoder` — PSA: mean-key block scores, progressive threshold selection with
                              fused attention.
* :class:`PRRDecoder`       — PRR: speculative attention over the EMA-predicted set P runs on a
                              second stream while scoring and top-K selection produce the true
                              set A; the repair pass adds A \\ P and drops P \\ A.
"""

from __future__ import annotations

import math

import torch

from . import binding as B


class Cache:
    """A paged bf16 KV cache on the GPU plus its descriptor."""

    def __init__(self, k_pages, v_pages, page_table, seq_lens, num_q_heads: int,
                 head_is_streaming=None):
        self.k_pages, self.v_pages = k_pages, v_pages
        self.page_table, self.seq_lens = page_table, seq_lens
        self.head_is_streaming = head_is_streaming
        self.num_q_heads = num_q_heads
        self.device = k_pages.device
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.kv = B.paged_kv(k_pages, v_pages, page_table, seq_lens, num_q_heads,
                             head_is_streaming, self.status)
        P, self.num_kv_heads, self.page_size, self.head_dim = k_pages.shape
        self.num_phys_pages = P
        self.batch, self.max_pages = page_table.shape
        self.group = num_q_heads // self.num_kv_heads
        self.rows = self.batch * self.num_kv_heads

    @classmethod
    def from_inputs(cls, inputs: dict, device="cuda") -> "Cache":
        w = inputs["workload"]
        t = {k: inputs[k].to(device) for k in ("k_pages", "v_pages", "page_table", "seq_lens",
                                                "head_is_streaming")}
        hs = t["head_is_streaming"] if w.streaming_kv_heads else None
        return cls(t["k_pages"], t["v_pages"], t["page_table"], t["seq_lens"], w.num_q_heads, hs)

    def append(self, k_new, v_new, metas=(), stream=None):
        """Decode-time append of one token per request (K and V bf16 ``[B][Hkv][D]``): advances
        ``seq_lens``, writes the token into its page and recomputes that page of every
        ``(kind, logical_page, meta)`` buffer in ``metas``.  The page table must already map the
        new position (a token that starts a page needs its page assigned first)."""
        self.seq_lens.add_(1)
        if not metas:
            B.dsa_append_kv(self.kv, k_new, v_new, stream=stream)
        for kind, lp, meta in metas:
            B.dsa_append_kv(self.kv, k_new, v_new, kind, lp, meta, stream)

    def kv8(self, stream=None):
        """The pools as KV8 blocks (e4m3 rows with one fp32 scale each, one contiguous block per
        (physical page, KV head)): a uint8 tensor; ``binding.kv8_unpack`` gives its parts."""
        buf = torch.empty(B.dsa_kv8_bytes(self.kv), dtype=torch.uint8, device=self.device)
        B.dsa_quantize_kv8(self.kv, buf, stream)
        return buf

    def kv4(self, stream=None):
        """The pools as KV4 blocks (4-bit integer rows with one fp32 scale each, one contiguous
        block per (physical page, KV head)): a uint8 tensor; ``binding.kv4_unpack`` gives its
        parts."""
        buf = torch.empty(B.dsa_kv4_bytes(self.kv), dtype=torch.uint8, device=self.device)
        B.dsa_quantize_kv4(self.kv, buf, stream)
        return buf

    def meta_buffer(self, kind: int, logical_page: int) -> torch.Tensor:
        g = self.page_size // logical_page
        if kind == B.DSA_META_MINMAX:
            return torch.zeros((self.num_phys_pages, self.num_kv_heads, g, self.head_dim, 2),
                               dtype=torch.bfloat16, device=self.device)
        return torch.zeros((self.num_phys_pages, self.num_kv_heads, g, self.head_dim),
                           dtype=torch.float32, device=self.device)

    def result_views(self):
        """(O, m, l, result): the three outputs as views of one contiguous fp32 buffer
        (``result``), so that a step's whole result reaches the host in one copy; each view starts
        on a 16-byte boundary."""
        nh = self.batch * self.num_q_heads
        nh4 = (nh + 3) // 4 * 4
        buf = torch.zeros(nh * self.head_dim + 2 * nh4, dtype=torch.float32, device=self.device)
        o = buf[:nh * self.head_dim].view(self.batch, self.num_q_heads, self.head_dim)
        m = buf[nh * self.head_dim:nh * self.head_dim + nh].view(self.batch, self.num_q_heads)
        l = buf[nh * self.head_dim + nh4:nh * self.head_dim + nh4 + nh].view(self.batch,
                                                                           self.num_q_heads)
        return o, m, l, buf

    def outputs(self):
        o, m, l, _ = self.result_views()
        return o, m, l


class TopKDecoder:
    def __init__(self, cache: Cache, k: int, logical_page: int | None = None,
                 meta_kind: int = B.DSA_META_MINMAX, scale: float | None = None):
        c = cache
        self.cache, self.k = c, k
        self.lp = logical_page or c.page_size
        self.kind = meta_kind
        self.scale = scale if scale is not None else 1.0 / math.sqrt(c.head_dim)
        self.meta = c.meta_buffer(meta_kind, self.lp)
        self.stride = c.max_pages * (c.page_size // self.lp)
        self.scores = torch.empty((c.batch, c.num_kv_heads, self.stride), dtype=torch.float32,
                                  device=c.device)
        self.idx = torch.empty((c.batch, c.num_kv_heads, max(1, k)), dtype=torch.int32,
                               device=c.device)
        self.count = torch.empty((c.batch, c.num_kv_heads), dtype=torch.int32, device=c.device)
        self.out, self.m, self.l, self.result = c.result_views()
        ws = B.dsa_sparse_decode_attn_workspace_size(c.kv, self.idx.shape[-1])
        self.workspace = torch.zeros(max(16, ws), dtype=torch.uint8, device=c.device)

    def build_meta(self, stream=None):
        B.dsa_build_page_meta(self.cache.kv, self.kind, self.lp, self.meta, stream)

    def append(self, k_new, v_new, stream=None):
        """Appends one decoded token per request, keeping this decoder's metadata current."""
        self.cache.append(k_new, v_new, [(self.kind, self.lp, self.meta)], stream)

    def use_kv8(self, stream=None):
        """Attends over KV8 pages from now on (the pools are quantised once, here); selection is
        unchanged (it reads the metadata)."""
        c = self.cache
        self.kv8 = c.kv8(stream)
        ws = B.dsa_sparse_decode_attn_kv8_workspace_size(c.kv, self.idx.shape[-1])
        self.kv8_workspace = torch.zeros(max(16, ws), dtype=torch.uint8, device=c.device)
        self.kv4 = None
        return self

    def use_kv4(self, stream=None):
        """Attends over KV4 pages from now on (the pools are quantised once, here)."""
        c = self.cache
        self.kv4 = c.kv4(stream)
        ws = B.dsa_sparse_decode_attn_kv4_workspace_size(c.kv, self.idx.shape[-1])
        self.kv4_workspace = torch.zeros(max(16, ws), dtype=torch.uint8, device=c.device)
        self.kv8 = None
        return self

    def select(self, q, stream=None):
        c = self.cache
        B.dsa_score_pages(c.kv, q, self.meta, self.kind, self.lp, self.scores, stream)
        B.dsa_select_topk(self.scores, self.stride, self.k, self.idx, self.count, stream)

    def attend(self, q, stream=None):
        if getattr(self, "kv4", None) is not None:
            B.dsa_sparse_decode_attn_kv4(self.cache.kv, self.kv4, q, self.idx, self.count,
                                         self.scale, self.out, self.m, self.l,
                                         self.kv4_workspace, stream)
            return
        if getattr(self, "kv8", None) is not None:
            B.dsa_sparse_decode_attn_kv8(self.cache.kv, self.kv8, q, self.idx, self.count,
                                         self.scale, self.out, self.m, self.l,
                                         self.kv8_workspace, stream)
            return
        B.dsa_sparse_decode_attn(self.cache.kv, q, self.idx, self.count, self.scale, self.out,
                                 self.m, self.l, workspace=self.workspace, stream=stream)

    def step(self, q, stream=None):
        self.select(q, stream)
        self.attend(q, stream)
        return self.out, self.m, self.l


class HierDecoder:
    def __init__(self, cache: Cache, k_phys: int, logical_page: int, sink: int, local: int,
                 reuse: int = 4, scale: float | None = None, one_launch: bool = True):
        """``one_launch``: dense and streaming heads attend in one launch
        (``dsa_hybrid_decode_attn``); otherwise as two (``dsa_sparse_decode_attn`` then
        ``dsa_streaming_head_attn``)."""
        c = cache
        self.cache, self.k, self.lp = c, k_phys, logical_page
        self.one_launch = one_launch
        self.g = c.page_size // logical_page
        self.sink, self.local, self.reuse = sink, local, reuse
        self.scale = scale if scale is not None else 1.0 / math.sqrt(c.head_dim)
        self.meta = c.meta_buffer(B.DSA_META_MINMAX, logical_page)
        self.stride = c.max_pages * self.g
        self.scores = torch.empty((c.batch, c.num_kv_heads, self.stride), dtype=torch.float32,
                                  device=c.device)
        self.idx = torch.empty((c.batch, c.num_kv_heads, max(1, k_phys)), dtype=torch.int32,
                               device=c.device)
        self.count = torch.empty((c.batch, c.num_kv_heads), dtype=torch.int32, device=c.device)
        self.out, self.m, self.l, self.result = c.result_views()
        ws = B.dsa_sparse_decode_attn_workspace_size(c.kv, self.idx.shape[-1])
        self.workspace = torch.zeros(max(16, ws), dtype=torch.uint8, device=c.device)

    def build_meta(self, stream=None):
        B.dsa_build_page_meta(self.cache.kv, B.DSA_META_MINMAX, self.lp, self.meta, stream)

    def append(self, k_new, v_new, stream=None):
        """Appends one decoded token per request, keeping this decoder's metadata current."""
        self.cache.append(k_new, v_new, [(B.DSA_META_MINMAX, self.lp, self.meta)], stream)

    def select(self, q, stream=None):
        c = self.cache
        B.dsa_score_pages(c.kv, q, self.meta, B.DSA_META_MINMAX, self.lp, self.scores, stream)
        B.dsa_select_hier(self.scores, self.stride, self.g, self.k, self.idx, self.count, stream)

    def step(self, q, t: int, stream=None):
        """Decode step t: selection runs when t is a multiple of the reuse interval (LServe §4.3),
        otherwise the previous selection is reused with this step's query."""
        c = self.cache
        if t % self.reuse == 0:
            self.select(q, stream)
        self.attend(q, stream)
        return self.out, self.m, self.l

    def attend(self, q, stream=None):
        c = self.cache
        if c.head_is_streaming is not None and self.one_launch:
            B.dsa_hybrid_decode_attn(c.kv, q, self.idx, self.count, self.sink, self.local,
                                     self.scale, self.out, self.m, self.l, self.workspace, stream)
            return
        B.dsa_sparse_decode_attn(c.kv, q, self.idx, self.count, self.scale, self.out, self.m,
                                 self.l, workspace=self.workspace, stream=stream)
        if c.head_is_streaming is not None:
            B.dsa_streaming_head_attn(c.kv, q, self.sink, self.local, self.scale, self.out,
                                      self.m, self.l, stream)


class ThresholdDecoder:
    def __init__(self, cache: Cache, tau: float, cap: int, use_nleft: bool = False,
                 scale: float | None = None):
        c = cache
        self.cache, self.tau, self.cap = c, tau, cap
        self.flags = B.DSA_PSA_NLEFT if use_nleft else 0
        self.scale = scale if scale is not None else 1.0 / math.sqrt(c.head_dim)
        self.meta = c.meta_buffer(B.DSA_META_MEAN, c.page_size)
        self.stride = c.max_pages
        self.scores = torch.empty((c.batch, c.num_kv_heads, self.stride), dtype=torch.float32,
                                  device=c.device)
        self.idx = torch.empty((c.batch, c.num_kv_heads, cap), dtype=torch.int32, device=c.device)
        self.count = torch.empty((c.batch, c.num_kv_heads), dtype=torch.int32, device=c.device)
        self.out, self.m, self.l, self.result = c.result_views()

    def build_meta(self, stream=None):
        B.dsa_build_page_meta(self.cache.kv, B.DSA_META_MEAN, self.cache.page_size, self.meta,
                              stream)

    def append(self, k_new, v_new, stream=None):
        """Appends one decoded token per request, keeping this decoder's metadata current."""
        self.cache.append(k_new, v_new, [(B.DSA_META_MEAN, self.cache.page_size, self.meta)],
                          stream)

    def step(self, q, stream=None):
        c = self.cache
        B.dsa_score_pages(c.kv, q, self.meta, B.DSA_META_MEAN, c.page_size, self.scores, stream)
        B.dsa_select_threshold(c.kv, q, self.scores, self.tau, self.cap, self.scale, self.idx,
                               self.count, self.out, self.m, self.l, self.flags, stream)
        return self.out, self.m, self.l


class PRRDecoder:
    """Predict, reuse and repair over top-K block selection (PRR §3.1-§3.4, fixed budget).

    With ``fused`` (the default) step t >= 1 is one ``dsa_prr_step`` launch: scoring with the EMA
    update and the speculative pass over P_t on most SMs, the selections of A_t and P_{t+1}, the
    repair and the merge on others, each waiting only for its own row's counters.  Otherwise the same
    library calls run as separate launches on three streams: the speculative pass over P_t on
    ``side``; scoring, top-K selection and the repair/merge on the caller's stream; the EMA update
    (which needs only this step's scores) on ``ema_stream``.  Either way P_{t+1} goes into the
    other half of a double-buffered list so that it never races the readers of P_t.
    """

    def __init__(self, cache: Cache, k: int, k_pred: int, alpha: float, beta: float,
                 gamma: float, superset: bool = False, scale: float | None = None,
                 two_streams: bool = True, fused: bool = True):
        c = cache
        self.cache, self.k, self.k_pred = c, k, k_pred
        self.alpha, self.beta, self.gamma = alpha, beta, gamma
        self.superset = superset
        self.scale = scale if scale is not None else 1.0 / math.sqrt(c.head_dim)
        self.meta = c.meta_buffer(B.DSA_META_MINMAX, c.page_size)
        self.stride = c.max_pages
        dev = c.device
        self.scores = torch.empty((c.batch, c.num_kv_heads, self.stride), dtype=torch.float32,
                                  device=dev)
        self.ell = torch.zeros_like(self.scores)
        self.trend = torch.zeros_like(self.scores)
        self.pred = torch.empty_like(self.scores)
        self.idx = torch.empty((c.batch, c.num_kv_heads, k), dtype=torch.int32, device=dev)
        self.count = torch.empty((c.batch, c.num_kv_heads), dtype=torch.int32, device=dev)
        self.spec_bufs = [torch.full((c.batch, c.num_kv_heads, k_pred), -1, dtype=torch.int32,
                                     device=dev) for _ in range(2)]
        self.spec_counts = [torch.zeros((c.batch, c.num_kv_heads), dtype=torch.int32, device=dev)
                            for _ in range(2)]
        self.partials = torch.empty((c.batch, c.num_kv_heads, k_pred, c.group, B.RECORD_FLOATS),
                                    dtype=torch.float32, device=dev)
        self.out, self.m, self.l, self.result = c.result_views()
        ws = max(B.dsa_repair_merge_workspace_size(c.kv, k),
                 B.dsa_sparse_decode_attn_workspace_size(c.kv, k))
        self.workspace = torch.zeros(max(16, ws), dtype=torch.uint8, device=dev)
        self.side = torch.cuda.Stream(device=dev) if two_streams else None
        self.ema_stream = torch.cuda.Stream(device=dev) if two_streams else None
        self.fused = fused
        # the fused step's workspace: its counters are zero before the first call and left zero
        # by each call
        self.step_workspace = torch.zeros(B.dsa_prr_step_workspace_size(c.kv), dtype=torch.uint8,
                                          device=dev)
        self.t = 0

    def calibrate(self, traj, stream=None):
        """PRR §3.2: rates the 80-point (alpha, beta, gamma) grid on a trajectory of true score
        vectors ``traj`` fp32 ``[steps][B][Hkv][stride]`` (e.g. scored during prefill) with
        ``dsa_calibrate_ema`` and adopts, for every row, the point that wins for most rows (ties to
        the lower point).  Returns (H ``[rows][80]``, best ``[rows]``)."""
        c = self.cache
        steps = traj.shape[0]
        t3 = traj.reshape(steps, c.batch * c.num_kv_heads, traj.shape[-1])
        rows = t3.shape[1]
        H = torch.empty((rows, B.CALIB_POINTS), dtype=torch.float32, device=c.device)
        best = torch.empty(rows, dtype=torch.int32, device=c.device)
        need = B.dsa_calibrate_ema_workspace_size(steps, rows, c.max_pages, self.k)
        ws = getattr(self, "calib_workspace", None)
        if ws is None or ws.numel() < need:
            self.calib_workspace = torch.zeros(need, dtype=torch.uint8, device=c.device)
        B.dsa_calibrate_ema(t3, c.max_pages, self.k, self.k_pred, H, best, self.calib_workspace,
                            stream)
        votes = torch.bincount(best.long(), minlength=B.CALIB_POINTS)
        self.alpha, self.beta, self.gamma = B.calibration_point(int(torch.argmax(votes)))
        return H, best

    def host_result(self):
        """Moves (O, m, l) into one page-locked host buffer that the fused step writes directly
        (no device-to-host copy); a fused step t >= 1 also accepts a page-locked host query.  The
        other steps (t = 0, or ``fused=False``) take device tensors only and refuse host ones."""
        o, m, l, buf = self.cache.result_views()  # the same layout, on the host
        pinned = torch.zeros(buf.shape, dtype=buf.dtype, pin_memory=True)
        n_o, n_h = o.numel(), m.numel()
        n_h4 = (buf.numel() - n_o) // 2
        self.result = pinned
        self.out = pinned[:n_o].view(o.shape)
        self.m = pinned[n_o:n_o + n_h].view(m.shape)
        self.l = pinned[n_o + n_h4:n_o + n_h4 + n_h].view(l.shape)
        return self

    @property
    def spec_idx(self):
        """The speculative set P the next step will use."""
        return self.spec_bufs[self.t % 2]

    @property
    def spec_count(self):
        return self.spec_counts[self.t % 2]

    def build_meta(self, stream=None):
        B.dsa_build_page_meta(self.cache.kv, B.DSA_META_MINMAX, self.cache.page_size, self.meta,
                              stream)

    def append(self, k_new, v_new, stream=None):
        """Appends one decoded token per request, keeping the metadata current.  The score rows
        and the predictor state already span the page table (stride = max pages), so a page that
        opens later needs nothing else: it gets a score once it holds a token, and the predictor
        treats it as fresh (level = its score, trend 0)."""
        c = self.cache
        c.append(k_new, v_new, [(B.DSA_META_MINMAX, c.page_size, self.meta)], stream)

    # ---- stages (one or two library calls each), exposed so a caller can time them one by one
    def stage_score(self, q, stream=None):
        c = self.cache
        B.dsa_score_pages(c.kv, q, self.meta, B.DSA_META_MINMAX, c.page_size, self.scores, stream)

    def stage_select(self, stream=None):
        B.dsa_select_topk(self.scores, self.stride, self.k, self.idx, self.count, stream)

    def stage_spec(self, q, buf: int = 0, stream=None):
        B.dsa_sparse_decode_attn(self.cache.kv, q, self.spec_bufs[buf], self.spec_counts[buf],
                                 self.scale, page_partials=self.partials, stream=stream)

    def stage_repair(self, q, buf: int = 0, stream=None):
        B.dsa_repair_merge(self.cache.kv, q, self.spec_bufs[buf], self.spec_counts[buf],
                           self.partials, self.idx, self.count, self.scale, self.out, self.m,
                           self.l, self.workspace, superset=self.superset, stream=stream)

    def stage_ema(self, mode=B.DSA_EMA_UPDATE, buf: int = 1, stream=None):
        B.dsa_ema_predict_update(self.scores, self.stride, self.ell, self.trend, mode, self.alpha,
                                 self.beta, self.gamma, self.pred, self.k_pred,
                                 self.spec_bufs[buf], self.spec_counts[buf], stream)

    def step(self, q):
        """One decode step with query q (bf16 [B][Hq][D]); returns (out, m, l)."""
        c = self.cache
        main = torch.cuda.current_stream(c.device)
        cur, nxt = self.t % 2, (self.t + 1) % 2
        if self.t == 0:
            self.stage_score(q, main)
            self.stage_select(main)
            B.dsa_sparse_decode_attn(c.kv, q, self.idx, self.count, self.scale, self.out, self.m,
                                     self.l, workspace=self.workspace, stream=main)
            self.stage_ema(B.DSA_EMA_INIT, nxt, main)
        elif self.fused:
            B.dsa_prr_step(c.kv, q, self.meta, self.scores, self.ell, self.trend, self.alpha,
                           self.beta, self.gamma, self.spec_bufs[cur], self.spec_counts[cur],
                           self.partials, self.idx, self.count, self.spec_bufs[nxt],
                           self.spec_counts[nxt], self.scale, self.out, self.m, self.l,
                           self.step_workspace, pred=self.pred, superset=self.superset,
                           stream=main)
        elif self.side is None:
            self.stage_score(q, main)
            self.stage_select(main)
            self.stage_ema(B.DSA_EMA_UPDATE, nxt, main)
            self.stage_spec(q, cur, main)
            self.stage_repair(q, cur, main)
        else:
            # speculative attention over P_t, concurrent with scoring and selection
            self.side.wait_stream(main)
            self.stage_spec(q, cur, self.side)
            self.stage_score(q, main)
            # the EMA needs only this step's scores: it runs beside selection and repair
            self.ema_stream.wait_stream(main)
            self.stage_ema(B.DSA_EMA_UPDATE, nxt, self.ema_stream)
            self.stage_select(main)
            main.wait_stream(self.side)
            self.stage_repair(q, cur, main)
            main.wait_stream(self.ema_stream)
        self.t += 1
        return self.out, self.m, self.l
