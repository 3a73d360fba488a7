"""Comparison rules shared by the GPU parity tests (test-side only; may use the oracle).

* Selected page sets are exact, except pages whose float64 oracle score lies within 1e-5 of the
  cut-off score (relative); the GPU still returns exactly the budgeted count.
* Outputs (O, m, l) pass when |gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise (fp32
  accumulation against float64).
* When a selection differs from the oracle's only inside the exemption, the GPU's set is checked
  to be a valid selection and the outputs are compared with the oracle's attention over that set.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle as O

ATOL, RTOL = 2e-3, 1e-2
TIE_REL = 1e-5


def f64(t) -> np.ndarray:
    return O.to_f64(t)


def row_tokens(pool, table, L: int, b: int, h: int) -> np.ndarray:
    """float64 ``[L][D]`` rows of request b / KV head h, gathered through the page table in one
    device-side index (same result as ``oracle.request_tokens``, faster for large rows)."""
    p = pool.shape[2]
    npages = -(-L // p)
    phys = table[b, :npages].long()
    rows = pool[phys, h].reshape(npages * p, pool.shape[3])[:L]
    return rows.double().cpu().numpy()


def assert_close(got, ref, what: str):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    g = np.where(both_inf, 0.0, got)
    r = np.where(both_inf, 0.0, ref)
    err = np.abs(g - r)
    bad = ~(err <= ATOL + RTOL * np.abs(r))
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu {got[i]!r} vs oracle {ref[i]!r}")


def assert_outputs(out, m, l, ref, what: str):
    Oref, mref, lref = ref
    assert_close(out, Oref, what + " O")
    assert_close(m, mref, what + " m")
    assert_close(l, lref, what + " l")


def check_topk(gpu_sel, scores64, k: int, what: str = "") -> bool:
    """Asserts the GPU's top-k set equals the oracle's up to near-ties at the cut-off.
    Returns True when the sets are identical."""
    gpu_sel = [int(x) for x in gpu_sel]
    ref = O.select_topk(scores64, k)
    assert len(set(gpu_sel)) == len(gpu_sel), f"{what}: duplicate pages {gpu_sel}"
    assert len(gpu_sel) == len(ref), f"{what}: {len(gpu_sel)} selected, oracle {len(ref)}"
    assert gpu_sel == sorted(gpu_sel), f"{what}: selection not ascending"
    if set(gpu_sel) == set(ref):
        return True
    ranked = O.rank_pages(scores64)
    cut = scores64[ranked[k - 1]]
    tol = TIE_REL * abs(cut)
    for j in set(gpu_sel) ^ set(ref):
        assert abs(scores64[j] - cut) <= tol, (
            f"{what}: page {j} (score {scores64[j]!r}) differs from the oracle's selection and is "
            f"not within {TIE_REL} of the cut-off {cut!r}")
    return False


def check_ranking(gpu_ranked, scores64, what: str = ""):
    """GPU visiting order vs the oracle ranking; adjacent entries may swap only when their float64
    scores are within TIE_REL of each other."""
    ref = O.rank_pages(scores64)[:len(gpu_ranked)]
    gpu_ranked = [int(x) for x in gpu_ranked]
    if gpu_ranked == ref:
        return True
    for a, b in zip(gpu_ranked, ref):
        if a != b:
            assert abs(scores64[a] - scores64[b]) <= TIE_REL * max(abs(scores64[a]), 1e-30), (
                f"{what}: rank differs at pages {a} vs {b}: scores {scores64[a]!r} {scores64[b]!r}")
    return False


def oracle_minmax_scores(keys64: np.ndarray, q_group, logical_page: int, stride: int):
    kmax, kmin = O.page_meta_minmax(keys64, logical_page)
    s = O.score_pages_minmax(O.representative_query(q_group), kmax, kmin)
    return O.pad_scores(s, stride)


def oracle_mean_scores(keys64: np.ndarray, q_group, block: int, stride: int):
    s = O.score_pages_mean(O.representative_query(q_group), O.page_meta_mean(keys64, block))
    return O.pad_scores(s, stride)


def to_cuda(inputs: dict) -> dict:
    out = dict(inputs)
    for k, v in inputs.items():
        if isinstance(v, torch.Tensor):
            out[k] = v.cuda()
    return out


def row_meta_minmax(pool, table, L: int, b: int, h: int, lp: int, chunk_pages: int = 1024):
    """Oracle kmax/kmin of one row, computed a chunk of pages at a time (chunks end on logical
    page boundaries, so the result equals ``oracle.page_meta_minmax`` over the whole row)."""
    p = pool.shape[2]
    npages = -(-L // p)
    kmax, kmin = [], []
    for c0 in range(0, npages, chunk_pages):
        c1 = min(npages, c0 + chunk_pages)
        phys = table[b, c0:c1].long()
        rows = pool[phys, h].reshape((c1 - c0) * p, pool.shape[3])[:L - c0 * p]
        a, z = O.page_meta_minmax(rows.double().cpu().numpy(), lp)
        kmax.append(a)
        kmin.append(z)
    return np.concatenate(kmax), np.concatenate(kmin)


def page_rows(pool, table, L: int, b: int, h: int, pages) -> np.ndarray:
    """float64 tokens of the listed page positions (clipped to L), concatenated in list order."""
    p = pool.shape[2]
    out = []
    for j in pages:
        n = min(p, L - int(j) * p)
        if n <= 0:
            continue
        out.append(pool[int(table[b, int(j)]), h, :n].double().cpu().numpy())
    if not out:
        return np.zeros((0, pool.shape[3]))
    return np.concatenate(out)


def attend_pages(q_group, kpool, vpool, table, L: int, b: int, h: int, pages, scale: float):
    """Oracle attention over the tokens of the listed pages (softmax attention is invariant to
    the order of its token set, so the pages' tokens are gathered compactly)."""
    K = page_rows(kpool, table, L, b, h, pages)
    V = page_rows(vpool, table, L, b, h, pages)
    return O.attend(q_group, K, V, np.arange(K.shape[0]), scale)
