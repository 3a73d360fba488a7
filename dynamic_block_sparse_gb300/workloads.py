"""Seeded synthetic decode workloads (inputs only; none of the method's arithmetic lives here).

Both the CUDA path and the CPU oracle are fed from these generators; neither imports the other.
The shapes follow the five long-context decode workloads the library is built for:

====  =======================  ==========================================================
idx   name                     shape
====  =======================  ==========================================================
0     tiny_topk                B1, 4 q / 1 KV head, D128, 4096 tokens, page 16, 8 hot pages,
                                kmax/kmin metadata, top-32 pages
1     llama3_8b_layer          B4, 32 q / 8 KV heads, 32K tokens, page 16, 64 hot pages per
                                KV head, top-256 pages (4096-token budget)
2     lserve_hier              B8, 32 q / 8 KV heads, 128K tokens, physical page 64 = 4
                                logical pages of 16, 64-page budget, KV heads 4..7 streaming
                                (64 sink + 256 local), selection reused over 4 steps, query
                                drift N(0, 0.1)
3     psa_threshold            B4, 32 q / 32 KV heads (MHA), 64K tokens, block 16, mean-key
                                metadata, Zipf(1.1) block masses planted by key alignment,
                                tau 0.95, cap 1024 blocks
4     prr_512k                 B1, 32 q / 2 KV heads, 512K tokens, block 64, top-64 blocks,
                                |P| = floor(1.2 * 64) = 76, 16 steps, query random walk
                                N(0, 0.05), EMA alpha 0.6 beta 0.3 gamma 0.5
====  =======================  ==========================================================

Keys, values and queries are N(0, 1) rounded to bf16.  "Hot" pages add ``hot_scale * u`` to every
key of the page, with ``u`` the unit direction of the group's summed step-0 query.  The Zipf
workload gives the block of rank r (a seeded permutation per row) keys ``c_r u + N(0, 1)`` with
``c_r = -(sqrt(D) / |q|) * s * ln r``, so that its expected attention mass falls as ``r^-s``.
Queries of later steps drift by adding ``drift * N(0, 1)`` to the fp32 query of the previous step,
then rounding to bf16.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: int
    page_size: int
    logical_page: int
    meta_kind: str                    # "minmax" | "mean"
    mode: str                         # "topk" | "hier" | "threshold" | "prr"
    k: int = 0                        # selected pages (topk / hier physical / PRR true set)
    cap: int = 0                      # PSA block cap
    tau: float = 0.0                  # PSA threshold
    hot_pages: int = 0
    hot_scale: float = 0.0
    zipf_s: float = 0.0
    streaming_kv_heads: tuple = ()
    sink: int = 0
    local: int = 0
    steps: int = 1
    reuse: int = 1                    # LServe reuse interval (selection every `reuse` steps)
    drift: float = 0.0
    delta: float = 0.0                # PRR speculation budget ratio
    alpha: float = 0.0
    beta: float = 0.0
    gamma: float = 0.0
    seed: int = 1000
    ragged: bool = False              # per-request lengths below seq_len (non-multiple of page)
    extra_phys_pages: int = 0         # unused pool pages (shuffled tables scatter into them)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def g(self) -> int:
        return self.page_size // self.logical_page

    @property
    def pages_per_seq(self) -> int:
        return -(-self.seq_len // self.page_size)

    @property
    def logical_per_seq(self) -> int:
        return -(-self.seq_len // self.logical_page)

    @property
    def num_phys_pages(self) -> int:
        return self.batch * self.pages_per_seq + self.extra_phys_pages

    @property
    def k_pred(self) -> int:
        return int(math.floor(self.delta * self.k + 1e-9))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def seq_lens(self) -> list[int]:
        if not self.ragged:
            return [self.seq_len] * self.batch
        out = []
        for b in range(self.batch):
            cut = (b * 7 + 3) % self.page_size if b > 0 else 0
            out.append(max(1, self.seq_len - cut - (b % 3) * self.page_size))
        return out

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def kv_bytes(self) -> int:
        return 2 * self.num_phys_pages * self.num_kv_heads * self.page_size * self.head_dim * 2


WORKLOADS: list[Workload] = [
    Workload("tiny_topk", 1, 4, 1, 128, 4096, 16, 16, "minmax", "topk", k=32,
             hot_pages=8, hot_scale=0.5, seed=1000),
    Workload("llama3_8b_layer", 4, 32, 8, 128, 32768, 16, 16, "minmax", "topk", k=256,
             hot_pages=64, hot_scale=0.5, seed=1001),
    Workload("lserve_hier", 8, 32, 8, 128, 131072, 64, 16, "minmax", "hier", k=64,
             streaming_kv_heads=(4, 5, 6, 7), sink=64, local=256, steps=4, reuse=4, drift=0.1,
             seed=1002),
    Workload("psa_threshold", 4, 32, 32, 128, 65536, 16, 16, "mean", "threshold",
             cap=1024, tau=0.95, zipf_s=1.1, seed=1003),
    Workload("prr_512k", 1, 32, 2, 128, 524288, 64, 64, "minmax", "prr", k=64, steps=16,
             drift=0.05, delta=1.2, alpha=0.6, beta=0.3, gamma=0.5, seed=1004),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def _gen(seed: int, tag: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tag)
    return g


def _randn(shape, gen, device, chunk_rows: int = 1 << 12) -> torch.Tensor:
    """N(0, 1) rounded to bf16, generated in slabs along dim 0 to bound fp32 temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    for s in range(0, n0, chunk_rows):
        e = min(n0, s + chunk_rows)
        out[s:e] = torch.randn((e - s,) + tuple(shape[1:]), generator=gen, device=device,
                               dtype=torch.float32).to(torch.bfloat16)
    return out


def make_inputs(w: Workload, device="cpu", shuffle_pages: bool = True) -> dict:
    """All tensors of one workload on ``device``.

    Returns a dict with ``k_pages``/``v_pages`` bf16 ``[P][Hkv][page][D]``, ``page_table`` int32
    ``[B][pages_per_seq]``, ``seq_lens`` int32 ``[B]``, ``q`` bf16 ``[steps][B][Hq][D]``,
    ``head_is_streaming`` uint8 ``[Hkv]`` and ``workload``.
    """
    device = torch.device(device)
    B, Hq, Hkv, D, p = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size
    P = w.num_phys_pages
    pps = w.pages_per_seq

    if shuffle_pages:
        perm = torch.randperm(P, generator=_gen(w.seed, 1, "cpu"))
        table = perm[:B * pps].reshape(B, pps)
    else:
        table = torch.arange(B * pps).reshape(B, pps)
    page_table = table.to(torch.int32).to(device)
    seq_lens = torch.tensor(w.seq_lens(), dtype=torch.int32, device=device)

    k_pages = _randn((P, Hkv, p, D), _gen(w.seed, 2, device), device)
    v_pages = _randn((P, Hkv, p, D), _gen(w.seed, 3, device), device)

    # queries: step 0 ~ N(0,1); later steps random-walk in fp32, each rounded to bf16 for use
    gq = _gen(w.seed, 4, device)
    q32 = torch.randn((B, Hq, D), generator=gq, device=device, dtype=torch.float32)
    qs = [q32.to(torch.bfloat16)]
    for _ in range(1, w.steps):
        q32 = q32 + w.drift * torch.randn((B, Hq, D), generator=gq, device=device,
                                          dtype=torch.float32)
        qs.append(q32.to(torch.bfloat16))
    q = torch.stack(qs, 0)

    G = w.group
    if w.hot_pages > 0:
        gh = _gen(w.seed, 5, "cpu")
        for b in range(B):
            npages = -(-int(seq_lens[b]) // p)
            for h in range(Hkv):
                direction = q[0, b, h * G:(h + 1) * G].float().sum(0)
                u = direction / direction.norm()
                pos = torch.randperm(npages, generator=gh)[:min(w.hot_pages, npages)]
                phys = page_table[b, pos.to(device)].long()
                blk = k_pages[phys, h].float() + w.hot_scale * u
                k_pages[phys, h] = blk.to(torch.bfloat16)

    if w.zipf_s > 0:
        gz = _gen(w.seed, 6, "cpu")
        for b in range(B):
            npages = -(-int(seq_lens[b]) // p)
            for h in range(Hkv):
                qh = q[0, b, h * G:(h + 1) * G].float().sum(0)
                qn = qh.norm()
                u = qh / qn
                rank = (torch.randperm(npages, generator=gz) + 1).to(device=device,
                                                                     dtype=torch.float32)
                c = -(math.sqrt(D) / qn) * w.zipf_s * torch.log(rank)
                phys = page_table[b, :npages].long()
                blk = k_pages[phys, h].float() + c[:, None, None] * u
                k_pages[phys, h] = blk.to(torch.bfloat16)

    streaming = torch.zeros(Hkv, dtype=torch.uint8)
    for h in w.streaming_kv_heads:
        if h < Hkv:
            streaming[h] = 1
    return dict(workload=w, k_pages=k_pages, v_pages=v_pages, page_table=page_table,
                seq_lens=seq_lens, q=q, head_is_streaming=streaming.to(device))


def oracle_scale(w: Workload) -> Workload:
    """A reduced version of a workload that the float64 oracle finishes in seconds, keeping its
    head layout, page geometry and selection mode, spanning several tiles, with ragged lengths."""
    if w.name == "tiny_topk":
        return w.replace(ragged=False)
    if w.name == "llama3_8b_layer":
        return w.replace(batch=2, num_q_heads=8, num_kv_heads=2, seq_len=2048 + 16 * 5, k=40,
                         hot_pages=6, ragged=True, extra_phys_pages=7)
    if w.name == "lserve_hier":
        return w.replace(batch=2, num_q_heads=16, num_kv_heads=4, seq_len=4096 + 64 * 3, k=12,
                         streaming_kv_heads=(2, 3), ragged=True, extra_phys_pages=5)
    if w.name == "psa_threshold":
        return w.replace(batch=2, num_q_heads=4, num_kv_heads=4, seq_len=4096 + 16 * 3, cap=64,
                         ragged=True, extra_phys_pages=3)
    if w.name == "prr_512k":
        return w.replace(seq_len=16384 + 64 * 2, k=16, steps=6, ragged=False, extra_phys_pages=4)
    raise KeyError(w.name)
