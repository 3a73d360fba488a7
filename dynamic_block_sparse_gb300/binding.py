"""ctypes binding of libdsa: the C-ABI entry points under the same names, taking torch tensors.

Argument marshalling only: every function passes device pointers, sizes and the current CUDA
stream to the library and raises :class:`DsaError` on a non-zero return code.  There is no
fallback: if ``libdsa.so`` is missing or cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re
import struct
from ctypes import c_float, c_int32, c_size_t, c_void_p

import torch

from . import build as _build

DSA_META_MINMAX, DSA_META_MEAN = 0, 1
DSA_EMA_INIT, DSA_EMA_UPDATE = 0, 1
DSA_PSA_NLEFT = 1
DSA_STATUS_BAD_PAGE, DSA_STATUS_OVERFLOW, DSA_STATUS_TIMEOUT = 1, 2, 4
RECORD_FLOATS = 132  # partial record: O[128], m, l, 0, 0

HEADER = os.path.join(_build.ROOT, "include", "dsa.h")


class DsaError(RuntimeError):
    def __init__(self, fn: str, rc: int, msg: str):
        super().__init__(f"{fn} failed with code {rc}: {msg}")
        self.rc = rc


class PagedKV(ctypes.Structure):
    _fields_ = [
        ("k_pages", c_void_p), ("v_pages", c_void_p), ("page_table", c_void_p),
        ("seq_lens", c_void_p), ("head_is_streaming", c_void_p), ("status", c_void_p),
        ("batch", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
        ("head_dim", c_int32), ("page_size", c_int32), ("max_pages_per_seq", c_int32),
        ("num_phys_pages", c_int32),
    ]


class PrrStepArgs(ctypes.Structure):
    """Mirror of ``dsa_prr_step_args``."""
    _fields_ = [
        ("q", c_void_p), ("meta", c_void_p), ("scores", c_void_p), ("stride", c_int32),
        ("ell", c_void_p), ("trend", c_void_p), ("alpha", c_float), ("beta", c_float),
        ("gamma", c_float), ("pred", c_void_p), ("spec_idx", c_void_p), ("spec_count", c_void_p),
        ("k_pred", c_int32), ("page_partials", c_void_p), ("idx", c_void_p),
        ("count", c_void_p), ("k", c_int32), ("next_idx", c_void_p), ("next_count", c_void_p),
        ("superset", c_int32), ("scale", c_float), ("out", c_void_p), ("m", c_void_p),
        ("l", c_void_p),
    ]


_P = c_void_p
_I = c_int32
_SIGNATURES = {
    "dsa_last_error": ([], ctypes.c_char_p),
    "dsa_version": ([], ctypes.c_char_p),
    "dsa_build_page_meta": ([_P, _I, _I, _P, _P], _I),
    "dsa_append_kv": ([_P, _P, _P, _I, _I, _P, _P], _I),
    "dsa_score_pages": ([_P, _P, _P, _I, _I, _P, _I, _P], _I),
    "dsa_select_topk": ([_P, _I, _I, _I, _I, _P, _I, _P, _P], _I),
    "dsa_select_hier": ([_P, _I, _I, _I, _I, _I, _P, _I, _P, _P], _I),
    "dsa_select_threshold": ([_P, _P, _P, _I, c_float, _I, _I, c_float, _P, _I, _P, _P, _P, _P,
                              _P], _I),
    "dsa_sparse_decode_attn": ([_P, _P, _P, _I, _P, c_float, _P, _P, _P, _P, _I, _P, c_size_t,
                                _P], _I),
    "dsa_sparse_decode_attn_workspace_size": ([_P, _I, _I], c_size_t),
    "dsa_sparse_decode_attn_noalloc": ([_P, _P, _P, _I, _P, c_float, _P, _P, _P, _I, _P], _I),
    "dsa_sparse_decode_attn_noalloc_max_bytes": ([], c_size_t),
    "dsa_repair_merge": ([_P, _P, _P, _I, _P, _P, _P, _I, _P, _I, c_float, _P, _P, _P, _P,
                          c_size_t, _P], _I),
    "dsa_repair_merge_workspace_size": ([_P, _I], c_size_t),
    "dsa_streaming_head_attn": ([_P, _P, _I, _I, c_float, _P, _P, _P, _P], _I),
    "dsa_hybrid_decode_attn": ([_P, _P, _P, _I, _P, _I, _I, c_float, _P, _P, _P, _P, c_size_t,
                                _P], _I),
    "dsa_quantize_kv8": ([_P, _P, _P], _I),
    "dsa_kv8_bytes": ([_P], c_size_t),
    "dsa_sparse_decode_attn_kv8": ([_P, _P, _P, _P, _I, _P, c_float, _P, _P, _P, _P, c_size_t,
                                    _P], _I),
    "dsa_sparse_decode_attn_kv8_workspace_size": ([_P, _I], c_size_t),
    "dsa_quantize_kv4": ([_P, _P, _P], _I),
    "dsa_kv4_bytes": ([_P], c_size_t),
    "dsa_sparse_decode_attn_kv4": ([_P, _P, _P, _P, _I, _P, c_float, _P, _P, _P, _P, c_size_t,
                                    _P], _I),
    "dsa_sparse_decode_attn_kv4_workspace_size": ([_P, _I], c_size_t),
    "dsa_ema_predict_update": ([_P, _I, _I, _I, _P, _P, _I, c_float, c_float, c_float, _P, _I,
                                _P, _I, _P, _P], _I),
    "dsa_merge_partials": ([_P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "dsa_calibrate_ema": ([_P, _I, _I, _I, _I, _I, _I, _P, _P, _P, c_size_t, _P], _I),
    "dsa_calibrate_ema_workspace_size": ([_I, _I, _I, _I], c_size_t),
    "dsa_prr_step": ([_P, _P, _P, c_size_t, _P], _I),
    "dsa_prr_step_workspace_size": ([_P], c_size_t),
    "dsa_prr_step_counter_bytes": ([_P], c_size_t),
}

_lib = None


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions ``include/dsa.h`` declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads libdsa.so (built in-tree by ``build()``) and declares every signature."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    return t.data_ptr()


def _io_ptr(t) -> int:
    """A CUDA tensor, or a page-locked host tensor the device reads or writes over the host link
    (the fused PRR step's query and result)."""
    if t.is_cuda or t.is_pinned():
        return t.data_ptr()
    raise ValueError("tensor must live on a CUDA device or in page-locked host memory")


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(name: str, rc: int) -> None:
    if rc != 0:
        raise DsaError(name, rc, load().dsa_last_error().decode())


def last_error() -> str:
    return load().dsa_last_error().decode()


def version() -> str:
    return load().dsa_version().decode()


def paged_kv(k_pages, v_pages, page_table, seq_lens, num_q_heads: int,
             head_is_streaming=None, status=None) -> PagedKV:
    """Descriptor of a paged cache; ``k_pages``/``v_pages`` are bf16 ``[P][Hkv][page][D]``."""
    P, Hkv, page, D = k_pages.shape
    assert k_pages.dtype == torch.bfloat16 and v_pages.shape == k_pages.shape
    assert page_table.dtype == torch.int32 and seq_lens.dtype == torch.int32
    kv = PagedKV()
    kv.k_pages = _ptr(k_pages)
    kv.v_pages = _ptr(v_pages)
    kv.page_table = _ptr(page_table)
    kv.seq_lens = _ptr(seq_lens)
    kv.head_is_streaming = _ptr(head_is_streaming)
    kv.status = _ptr(status)
    kv.batch = page_table.shape[0]
    kv.num_q_heads = num_q_heads
    kv.num_kv_heads = Hkv
    kv.head_dim = D
    kv.page_size = page
    kv.max_pages_per_seq = page_table.shape[1]
    kv.num_phys_pages = P
    return kv


def dsa_build_page_meta(kv: PagedKV, meta_kind: int, logical_page: int, meta, stream=None):
    _check("dsa_build_page_meta", load().dsa_build_page_meta(
        ctypes.byref(kv), meta_kind, logical_page, _ptr(meta), _stream(stream)))


def dsa_append_kv(kv: PagedKV, k_new, v_new, meta_kind: int = 0, logical_page: int = 0,
                  meta=None, stream=None):
    """Writes the token at position seq_lens[b] - 1 (already counted) of every request into the
    pools and recomputes its page's metadata in ``meta`` (if given)."""
    _check("dsa_append_kv", load().dsa_append_kv(
        ctypes.byref(kv), _ptr(k_new), _ptr(v_new), meta_kind, logical_page, _ptr(meta),
        _stream(stream)))


def dsa_score_pages(kv: PagedKV, q, meta, meta_kind: int, logical_page: int, scores,
                    stream=None):
    _check("dsa_score_pages", load().dsa_score_pages(
        ctypes.byref(kv), _ptr(q), _ptr(meta), meta_kind, logical_page, _ptr(scores),
        scores.shape[-1], _stream(stream)))


def dsa_select_topk(scores, n: int, k: int, idx, count, stream=None):
    rows = scores.numel() // scores.shape[-1]
    _check("dsa_select_topk", load().dsa_select_topk(
        _ptr(scores), rows, n, scores.shape[-1], k, _ptr(idx), idx.shape[-1], _ptr(count),
        _stream(stream)))


def dsa_select_hier(logical_scores, n_logical: int, g: int, k_phys: int, idx, count,
                    stream=None):
    rows = logical_scores.numel() // logical_scores.shape[-1]
    _check("dsa_select_hier", load().dsa_select_hier(
        _ptr(logical_scores), rows, n_logical, logical_scores.shape[-1], g, k_phys, _ptr(idx),
        idx.shape[-1], _ptr(count), _stream(stream)))


def dsa_select_threshold(kv: PagedKV, q, scores, tau: float, cap: int, scale: float, idx, count,
                         out, m, l, flags: int = 0, stream=None):
    _check("dsa_select_threshold", load().dsa_select_threshold(
        ctypes.byref(kv), _ptr(q), _ptr(scores), scores.shape[-1], tau, cap, flags, scale,
        _ptr(idx), idx.shape[-1], _ptr(count), _ptr(out), _ptr(m), _ptr(l), _stream(stream)))


def dsa_sparse_decode_attn_workspace_size(kv: PagedKV, idx_stride: int, num_splits: int = 0) -> int:
    return int(load().dsa_sparse_decode_attn_workspace_size(ctypes.byref(kv), idx_stride,
                                                            num_splits))


def dsa_sparse_decode_attn(kv: PagedKV, q, idx, count, scale: float, out=None, m=None, l=None,
                           page_partials=None, num_splits: int = 0, workspace=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("dsa_sparse_decode_attn", load().dsa_sparse_decode_attn(
        ctypes.byref(kv), _ptr(q), _ptr(idx), idx.shape[-1], _ptr(count), scale, _ptr(out),
        _ptr(m), _ptr(l), _ptr(page_partials), num_splits, _ptr(workspace), ws_bytes,
        _stream(stream)))


def dsa_sparse_decode_attn_noalloc(kv: PagedKV, q, idx, count, scale: float, out, m, l,
                                   num_splits: int = 0, stream=None):
    """dsa_sparse_decode_attn with the split records in the library's fixed device scratch (for
    callers that must not allocate); calls must not overlap on the GPU."""
    _check("dsa_sparse_decode_attn_noalloc", load().dsa_sparse_decode_attn_noalloc(
        ctypes.byref(kv), _ptr(q), _ptr(idx), idx.shape[-1], _ptr(count), scale, _ptr(out),
        _ptr(m), _ptr(l), num_splits, _stream(stream)))


def dsa_sparse_decode_attn_noalloc_max_bytes() -> int:
    return int(load().dsa_sparse_decode_attn_noalloc_max_bytes())


def dsa_repair_merge_workspace_size(kv: PagedKV, true_stride: int) -> int:
    return int(load().dsa_repair_merge_workspace_size(ctypes.byref(kv), true_stride))


def dsa_repair_merge(kv: PagedKV, q, spec_idx, spec_count, page_partials, true_idx, true_count,
                     scale: float, out, m, l, workspace, superset: bool = False, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_repair_merge", load().dsa_repair_merge(
        ctypes.byref(kv), _ptr(q), _ptr(spec_idx), spec_idx.shape[-1], _ptr(spec_count),
        _ptr(page_partials), _ptr(true_idx), true_idx.shape[-1], _ptr(true_count),
        1 if superset else 0, scale, _ptr(out), _ptr(m), _ptr(l), _ptr(workspace), ws_bytes,
        _stream(stream)))


def dsa_hybrid_decode_attn(kv: PagedKV, q, idx, count, sink: int, local: int, scale: float,
                           out, m, l, workspace, stream=None):
    """Dense heads over their selected pages and streaming heads over sink + local tokens, one
    launch."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_hybrid_decode_attn", load().dsa_hybrid_decode_attn(
        ctypes.byref(kv), _ptr(q), _ptr(idx), idx.shape[-1], _ptr(count), sink, local, scale,
        _ptr(out), _ptr(m), _ptr(l), _ptr(workspace), ws_bytes, _stream(stream)))


def dsa_kv8_bytes(kv: PagedKV) -> int:
    return int(load().dsa_kv8_bytes(ctypes.byref(kv)))


def dsa_quantize_kv8(kv: PagedKV, kv8, stream=None):
    """bf16 pools -> KV8 blocks (uint8 tensor of dsa_kv8_bytes(kv) bytes): per (physical page, KV
    head) the e4m3 K codes [p][128], V codes [p][128] (16-byte pieces XOR-permuted by the token
    slot mod 8), K scales fp32 [p], V scales fp32 [p]; ``kv8_unpack`` takes them apart."""
    _check("dsa_quantize_kv8", load().dsa_quantize_kv8(ctypes.byref(kv), _ptr(kv8),
                                                       _stream(stream)))


def kv8_unpack(kv8, num_phys_pages: int, num_kv_heads: int, page: int):
    """The parts of a KV8 buffer: (K codes, V codes) uint8 ``[P][Hkv][p][128]`` in dim order (the
    stored rows keep their 16-byte pieces XOR-permuted by the token slot mod 8) and (K scales, V
    scales) fp32 ``[P][Hkv][p]``."""
    blk = kv8.view(num_phys_pages, num_kv_heads, 264 * page)
    # piece c of slot r is stored at piece c ^ (r % 8); the permutation is its own inverse
    r = torch.arange(page, device=kv8.device).view(page, 1)
    c = torch.arange(8, device=kv8.device).view(1, 8)
    perm = (c ^ (r % 8)).view(1, 1, page, 8, 1).expand(num_phys_pages, num_kv_heads, page, 8, 16)

    def codes(part):
        rows = part.reshape(num_phys_pages, num_kv_heads, page, 8, 16)
        return torch.gather(rows, 3, perm).reshape(num_phys_pages, num_kv_heads, page, 128)

    kc = codes(blk[..., :128 * page])
    vc = codes(blk[..., 128 * page:256 * page])
    ks = blk[..., 256 * page:260 * page].contiguous().view(torch.float32)
    vs = blk[..., 260 * page:].contiguous().view(torch.float32)
    return kc, vc, ks, vs


def dsa_sparse_decode_attn_kv8_workspace_size(kv: PagedKV, idx_stride: int) -> int:
    return int(load().dsa_sparse_decode_attn_kv8_workspace_size(ctypes.byref(kv), idx_stride))


def dsa_sparse_decode_attn_kv8(kv: PagedKV, kv8, q, idx, count, scale: float, out, m, l,
                               workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_sparse_decode_attn_kv8", load().dsa_sparse_decode_attn_kv8(
        ctypes.byref(kv), _ptr(kv8), _ptr(q), _ptr(idx), idx.shape[-1], _ptr(count), scale,
        _ptr(out), _ptr(m), _ptr(l), _ptr(workspace), ws_bytes, _stream(stream)))


def dsa_kv4_bytes(kv: PagedKV) -> int:
    return int(load().dsa_kv4_bytes(ctypes.byref(kv)))


def dsa_quantize_kv4(kv: PagedKV, kv4, stream=None):
    """bf16 pools -> KV4 blocks (uint8 tensor of dsa_kv4_bytes(kv) bytes): per (physical page, KV
    head) the K code rows [p][64], V code rows [p][64] (offset-8 nibbles, two dims per byte; row
    of slot r stored at r ^ ((r >> 1) & 1)), K scales fp32 [p], V scales fp32 [p];
    ``kv4_unpack`` takes them apart."""
    _check("dsa_quantize_kv4", load().dsa_quantize_kv4(ctypes.byref(kv), _ptr(kv4),
                                                       _stream(stream)))


def kv4_unpack(kv4, num_phys_pages: int, num_kv_heads: int, page: int):
    """The parts of a KV4 buffer: (K rows, V rows) uint8 ``[P][Hkv][p][64]`` in token order (packed
    nibbles as stored) and (K scales, V scales) fp32 ``[P][Hkv][p]``."""
    blk = kv4.view(num_phys_pages, num_kv_heads, 136 * page)
    r = torch.arange(page, device=kv4.device)
    perm = r ^ ((r >> 1) & 1)  # its own inverse

    def rows(part):
        return part.reshape(num_phys_pages, num_kv_heads, page, 64)[:, :, perm, :]

    kc = rows(blk[..., :64 * page])
    vc = rows(blk[..., 64 * page:128 * page])
    ks = blk[..., 128 * page:132 * page].contiguous().view(torch.float32)
    vs = blk[..., 132 * page:].contiguous().view(torch.float32)
    return kc, vc, ks, vs


def dsa_sparse_decode_attn_kv4_workspace_size(kv: PagedKV, idx_stride: int) -> int:
    return int(load().dsa_sparse_decode_attn_kv4_workspace_size(ctypes.byref(kv), idx_stride))


def dsa_sparse_decode_attn_kv4(kv: PagedKV, kv4, q, idx, count, scale: float, out, m, l,
                               workspace, stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_sparse_decode_attn_kv4", load().dsa_sparse_decode_attn_kv4(
        ctypes.byref(kv), _ptr(kv4), _ptr(q), _ptr(idx), idx.shape[-1], _ptr(count), scale,
        _ptr(out), _ptr(m), _ptr(l), _ptr(workspace), ws_bytes, _stream(stream)))


def dsa_streaming_head_attn(kv: PagedKV, q, sink: int, local: int, scale: float, out, m, l,
                            stream=None):
    _check("dsa_streaming_head_attn", load().dsa_streaming_head_attn(
        ctypes.byref(kv), _ptr(q), sink, local, scale, _ptr(out), _ptr(m), _ptr(l),
        _stream(stream)))


def dsa_ema_predict_update(IS, n: int, ell, v, mode: int, alpha: float, beta: float,
                           gamma: float, pred=None, k_pred: int = 0, pred_idx=None,
                           pred_count=None, stream=None):
    rows = IS.numel() // IS.shape[-1]
    _check("dsa_ema_predict_update", load().dsa_ema_predict_update(
        _ptr(IS), rows, n, IS.shape[-1], _ptr(ell), _ptr(v), mode, alpha, beta, gamma,
        _ptr(pred), k_pred, _ptr(pred_idx), 0 if pred_idx is None else pred_idx.shape[-1],
        _ptr(pred_count), _stream(stream)))


CALIB_POINTS = 80


def calibration_point(c: int) -> tuple[float, float, float]:
    """(alpha, beta, gamma) of grid point c of dsa_calibrate_ema (alpha outermost, gamma
    innermost), as the fp32 values the kernel uses."""
    def f32(x: float) -> float:
        return struct.unpack("f", struct.pack("f", x))[0]

    # an fp32 constant times a small integer, rounded to fp32 (as the kernel computes it)
    return (f32(f32(0.2) * (1 + c // 20)), f32(f32(0.1) * (1 + (c // 4) % 5)),
            f32(f32(0.25) * (c % 4)))


def dsa_calibrate_ema_workspace_size(steps: int, rows: int, n: int, k: int) -> int:
    return int(load().dsa_calibrate_ema_workspace_size(steps, rows, n, k))


def dsa_calibrate_ema(traj, n: int, k: int, k_pred: int, H, best, workspace, stream=None):
    """``traj`` fp32 ``[steps][rows][stride]`` -> ``H`` fp32 ``[rows][80]`` and ``best`` int32
    ``[rows]`` (the winning grid point).  ``workspace``: dsa_calibrate_ema_workspace_size(steps,
    rows, n, k) bytes, zero-filled before its first use (each completed call leaves the part that
    must be zero zero-filled)."""
    steps, rows, stride = traj.shape
    assert H.shape[-1] == CALIB_POINTS
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_calibrate_ema", load().dsa_calibrate_ema(
        _ptr(traj), steps, rows, n, stride, k, k_pred, _ptr(H), _ptr(best), _ptr(workspace),
        ws_bytes, _stream(stream)))


def dsa_merge_partials(partials, out, m, l, stream=None):
    """``partials`` fp32 ``[rows][parts][G][132]`` -> ``out [rows*G][128]``, ``m``, ``l``."""
    rows, parts, G, rec = partials.shape
    assert rec == RECORD_FLOATS
    _check("dsa_merge_partials", load().dsa_merge_partials(
        _ptr(partials), rows, parts, G, 128, _ptr(out), _ptr(m), _ptr(l), _stream(stream)))


def dsa_prr_step_workspace_size(kv: PagedKV) -> int:
    return int(load().dsa_prr_step_workspace_size(ctypes.byref(kv)))


def dsa_prr_step_counter_bytes(kv: PagedKV) -> int:
    return int(load().dsa_prr_step_counter_bytes(ctypes.byref(kv)))


def dsa_prr_step(kv: PagedKV, q, meta, scores, ell, trend, alpha: float, beta: float,
                 gamma: float, spec_idx, spec_count, page_partials, idx, count, next_idx,
                 next_count, scale: float, out, m, l, workspace, pred=None,
                 superset: bool = False, stream=None):
    """One PRR decode step (scoring, top-k, speculation over P_t, EMA update with the selection
    of P_{t+1}, repair and merge) in one launch.  ``workspace`` must be zero-filled before its
    first use (each completed call leaves it zero-filled).  ``q`` and ``out``/``m``/``l`` may be
    page-locked host tensors: the kernel reads and writes them over the host link."""
    a = PrrStepArgs()
    a.q, a.meta, a.scores, a.stride = _io_ptr(q), _ptr(meta), _ptr(scores), scores.shape[-1]
    a.ell, a.trend = _ptr(ell), _ptr(trend)
    a.alpha, a.beta, a.gamma, a.pred = alpha, beta, gamma, _ptr(pred)
    a.spec_idx, a.spec_count, a.k_pred = _ptr(spec_idx), _ptr(spec_count), spec_idx.shape[-1]
    a.page_partials = _ptr(page_partials)
    a.idx, a.count, a.k = _ptr(idx), _ptr(count), idx.shape[-1]
    a.next_idx, a.next_count = _ptr(next_idx), _ptr(next_count)
    assert next_idx.shape[-1] == spec_idx.shape[-1]
    a.superset, a.scale = 1 if superset else 0, scale
    a.out, a.m, a.l = _io_ptr(out), _io_ptr(m), _io_ptr(l)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("dsa_prr_step", load().dsa_prr_step(ctypes.byref(kv), ctypes.byref(a), _ptr(workspace),
                                               ws_bytes, _stream(stream)))
