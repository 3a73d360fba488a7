"""CPU-only checks of the host side: the C-ABI library builds, loads and exports every symbol the
header declares; host-side argument validation answers without touching a GPU; the input
generator is deterministic and plants what it says; the replica timing reduction works across
processes (gloo)."""

import ctypes
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dynamic_block_sparse_gb300 import binding, build
    build.build()
    return binding.load()


def test_library_exports_every_header_function(lib):
    from dynamic_block_sparse_gb300 import binding, build
    names = binding.header_functions()
    assert len(names) >= 14
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in nm.splitlines() if ln.strip()}
    for n in names:
        assert n in exported, f"{n} declared in include/dsa.h but not exported"
        assert hasattr(lib, n)
    assert set(binding._SIGNATURES) == set(names), "binding signatures out of sync with the header"


def test_header_struct_layout_matches_binding(tmp_path):
    """Every field of the header's structs sits at the offset the ctypes mirror uses (a C
    program compiled against include/dsa.h prints the offsets)."""
    from dynamic_block_sparse_gb300 import binding
    assert ctypes.sizeof(binding.PagedKV) == 6 * 8 + 7 * 4 + 4  # 6 pointers, 7 int32, padding
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "dsa.h"', "int main(void) {"]
    for cname, cls in (("dsa_paged_kv", binding.PagedKV), ("dsa_prr_step_args", binding.PrrStepArgs)):
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True)
    got = dict(ln.split() for ln in subprocess.run([str(exe)], capture_output=True, text=True,
                                                    check=True).stdout.splitlines())
    for cname, cls in (("dsa_paged_kv", binding.PagedKV), ("dsa_prr_step_args", binding.PrrStepArgs)):
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for f, _ in cls._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(cls, f).offset, f"{cname}.{f}"


def test_version_and_empty_error(lib):
    assert b"sm_103a" in lib.dsa_version()
    assert lib.dsa_last_error() == b""


def test_host_validation_without_gpu(lib):
    from dynamic_block_sparse_gb300 import binding as B
    rc = lib.dsa_build_page_meta(None, 0, 16, None, None)
    assert rc == -1 and b"kv descriptor" in lib.dsa_last_error()
    kv = B.PagedKV()
    kv.k_pages = kv.v_pages = kv.page_table = kv.seq_lens = 4096
    kv.batch, kv.num_q_heads, kv.num_kv_heads = 1, 32, 2
    kv.head_dim, kv.page_size, kv.max_pages_per_seq, kv.num_phys_pages = 64, 64, 8, 8
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 64, 4096, None) == -3
    assert b"head_dim" in lib.dsa_last_error()
    kv.head_dim = 128
    kv.page_size = 24
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 24, 4096, None) == -3
    kv.page_size = 64
    kv.num_q_heads = 40
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 64, 4096, None) == -3    # G = 20 > 16
    kv.num_q_heads = 32
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 48, 4096, None) == -1    # lp does not divide
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 64, 4100, None) == -2    # misaligned meta
    kv.k_pages = 4104
    assert lib.dsa_build_page_meta(ctypes.byref(kv), 0, 64, 4096, None) == -2    # misaligned pool
    assert lib.dsa_select_topk(None, 2, 10, 10, 5, None, 5, None, None) == -1
    assert lib.dsa_select_topk(None, 0, 10, 10, 5, None, 5, None, None) == 0     # nothing to do
    assert lib.dsa_select_topk(4096, 1, 40000, 40000, 5, 4096, 5, 4096, None) == -3
    assert lib.dsa_ema_predict_update(4096, 1, 10, 10, 4096, 4096, 7, 0.6, 0.3, 0.5, None, 0,
                                      None, 0, None, None) == -1
    kv.k_pages = 4096
    assert lib.dsa_select_threshold(ctypes.byref(kv), 4096, 4096, 8, 1.5, 4, 0, 0.1, 4096, 4,
                                    4096, 4096, 4096, 4096, None) == -1          # tau > 1
    assert lib.dsa_sparse_decode_attn_workspace_size(ctypes.byref(kv), 64, 1) == 0
    assert lib.dsa_sparse_decode_attn_workspace_size(ctypes.byref(kv), 64, 4) == 2 * 4 * 16 * 132 * 4
    assert lib.dsa_repair_merge_workspace_size(ctypes.byref(kv), 64) == 2 * 16 * 16 * 132 * 4


def test_binding_refuses_cpu_tensors(lib):
    from dynamic_block_sparse_gb300 import binding as B
    with pytest.raises(ValueError, match="CUDA"):
        B.dsa_select_topk(torch.zeros(2, 8), 8, 2, torch.zeros((2, 2), dtype=torch.int32),
                          torch.zeros(2, dtype=torch.int32))


def test_append_kv_host_validation_without_gpu(lib):
    """dsa_append_kv rejects bad arguments on the host, before any CUDA call."""
    from dynamic_block_sparse_gb300 import binding as B
    kv = B.PagedKV()
    kv.k_pages = kv.v_pages = kv.page_table = kv.seq_lens = 4096
    kv.batch, kv.num_q_heads, kv.num_kv_heads = 2, 8, 2
    kv.head_dim, kv.page_size, kv.max_pages_per_seq, kv.num_phys_pages = 128, 64, 8, 16
    call = lambda k=8192, v=8192, kind=0, lp=16, meta=16384: lib.dsa_append_kv(
        ctypes.byref(kv), k, v, kind, lp, meta, None)
    assert call(k=0) == -1
    assert call(v=8200) == -2                                          # misaligned v_new
    assert call(kind=7) == -1
    assert call(lp=24) == -1 and b"divide" in lib.dsa_last_error()     # 24 does not divide 64
    assert call(meta=16392) == -2                                      # misaligned meta


def test_calibrate_ema_host_validation_without_gpu(lib):
    """dsa_calibrate_ema rejects bad arguments on the host, before any CUDA call."""
    p = 4096
    need = lib.dsa_calibrate_ema_workspace_size(8, 3, 500, 16)
    # counters, A_t counts and indices of every (step, row), predictor state of every (row, point)
    assert need == 16 + 96 + 8 * 3 * 16 * 4 + 3 * 80 * 2 * 500 * 4
    call = lambda steps=8, rows=3, n=500, stride=512, k=16, kp=20, ws=need: \
        lib.dsa_calibrate_ema(p, steps, rows, n, stride, k, kp, p * 2, p * 3, p * 4, ws, None)
    assert lib.dsa_calibrate_ema(p, 8, 0, 500, 512, 16, 20, p, p, p, 0, None) == 0  # no rows
    assert call(steps=0) == -1 and b"steps" in lib.dsa_last_error()
    assert call(n=600) == -1                                           # n > stride
    assert call(n=20000, stride=20000) == -3                           # predictor state too big
    assert call(k=300) == -3 and call(kp=0) == -1
    assert call(ws=need - 1) == -5
    assert lib.dsa_calibrate_ema(0, 8, 3, 500, 512, 16, 20, p, p, p, need, None) == -1  # NULL traj


def test_prr_step_host_validation_without_gpu(lib):
    """dsa_prr_step rejects bad arguments on the host, before any CUDA call."""
    from dynamic_block_sparse_gb300 import binding as B
    kv = B.PagedKV()
    kv.k_pages = kv.v_pages = kv.page_table = kv.seq_lens = 4096
    kv.batch, kv.num_q_heads, kv.num_kv_heads = 1, 32, 2
    kv.head_dim, kv.page_size, kv.max_pages_per_seq, kv.num_phys_pages = 128, 64, 64, 64
    a = B.PrrStepArgs()
    for i, f in enumerate(("q", "meta", "scores", "ell", "trend", "spec_idx", "spec_count",
                           "page_partials", "idx", "count", "next_count", "out", "m", "l")):
        setattr(a, f, 4096 * (1 + i))
    a.stride, a.k, a.k_pred, a.scale = 64, 8, 10, 0.1
    ws = 1 << 20
    call = lambda: lib.dsa_prr_step(ctypes.byref(kv), ctypes.byref(a), ws, 1 << 20, None)
    assert call() == -1 and b"NULL" in lib.dsa_last_error()          # next_idx missing
    a.next_idx = a.spec_idx
    assert call() == -1 and b"alias" in lib.dsa_last_error()
    a.next_idx = 4096 * 99
    a.stride = 32
    assert call() == -1 and b"stride" in lib.dsa_last_error()        # < max_pages_per_seq
    a.stride = 64
    a.k = 300
    assert call() == -3
    a.k = 8
    a.q = 4100
    assert call() == -2                                               # misaligned q
    a.q = 4096
    need = lib.dsa_prr_step_workspace_size(ctypes.byref(kv))
    # 2 rows: the exit word and two per-row counter arrays (16 bytes each); then the per-row
    # candidate hints (16 bytes), one 128-byte candidate line per row for each of up to 160 worker
    # CTAs, and the new predictions (max_pages_per_seq = 64 floats per row)
    counters = 16 + 2 * 16
    assert lib.dsa_prr_step_counter_bytes(ctypes.byref(kv)) == counters
    assert need == counters + 16 + 2 * 160 * 128 + 2 * 64 * 4
    assert lib.dsa_prr_step(ctypes.byref(kv), ctypes.byref(a), ws, need - 1, None) == -5
    kv.head_is_streaming = 4096
    assert call() == -3 and b"streaming" in lib.dsa_last_error()
    assert lib.dsa_prr_step(ctypes.byref(kv), None, ws, 1 << 20, None) == -1
    assert lib.dsa_prr_step_workspace_size(None) == 0


def test_generator_is_deterministic_and_plants_hot_pages():
    from dynamic_block_sparse_gb300.workloads import oracle_scale, BY_NAME, make_inputs
    w = oracle_scale(BY_NAME["llama3_8b_layer"])
    a, b = make_inputs(w), make_inputs(w)
    for k in ("k_pages", "v_pages", "page_table", "seq_lens", "q"):
        assert torch.equal(a[k], b[k])
    assert a["k_pages"].dtype == torch.bfloat16
    assert sorted(a["page_table"].flatten().tolist()) == sorted(set(a["page_table"].flatten().tolist()))
    # hot pages: mean key projection on the query direction is ~hot_scale above the rest
    G = w.group
    q = a["q"][0, 0, :G].float().sum(0)
    u = q / q.norm()
    L = int(a["seq_lens"][0])
    proj = []
    for j in range(-(-L // w.page_size)):
        proj.append(float(a["k_pages"][int(a["page_table"][0, j]), 0].float().mean(0) @ u))
    proj = np.sort(np.array(proj))[::-1]
    assert proj[: w.hot_pages].mean() > proj[w.hot_pages:].mean() + 0.3


def test_zipf_workload_masses_follow_rank():
    from dynamic_block_sparse_gb300.workloads import oracle_scale, BY_NAME, make_inputs
    w = oracle_scale(BY_NAME["psa_threshold"]).replace(batch=1, num_q_heads=1, num_kv_heads=1)
    a = make_inputs(w)
    q = a["q"][0, 0, 0].float()
    L = int(a["seq_lens"][0])
    logits = []
    for j in range(-(-L // 16)):
        k = a["k_pages"][int(a["page_table"][0, j]), 0].float()
        logits.append(float((k @ q).mean() / math.sqrt(128)))
    logits = np.sort(np.array(logits))[::-1]
    r = np.arange(1, len(logits) + 1)
    slope = np.polyfit(np.log(r[:200]), logits[:200], 1)[0]
    assert -1.4 < slope < -0.8           # mean logit of rank r falls like -1.1 ln r


def test_bench_byte_accounting():
    sys.path.insert(0, ROOT)
    import bench
    from dynamic_block_sparse_gb300.workloads import BY_NAME
    w = BY_NAME["prr_512k"]
    total, true_set, parts = bench.prr_bytes(w, 8192, 152, 4)
    assert parts["meta"] == 2 * 8192 * 512
    assert parts["kv"] == 156 * 64 * 512
    assert true_set == 2 * 8192 * 512 + 2 * 64 * 64 * 512
    # the partial records stay in L2: reported apart, not counted
    assert total == parts["meta"] + parts["kv"] + parts["aux"]
    assert parts["records_l2"] == 156 * 16 * 132 * 4


def _replica_worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    dist.barrier()
    v = bench.max_over_ranks(1.0 + rank * 2.5)
    with open(out + f".{rank}", "w") as f:
        json.dump(v, f)
    dist.destroy_process_group()


def test_replica_timing_takes_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp
    port = 29500 + (os.getpid() % 1000)
    out = str(tmp_path / "r")
    mp.spawn(_replica_worker, args=(2, port, out), nprocs=2, join=True)
    vals = [json.load(open(out + f".{r}")) for r in range(2)]
    assert vals == [3.5, 3.5]


def test_kv8_unpack_reads_the_documented_layout():
    """A KV8 buffer written byte by byte from the layout the header documents (per (page, KV
    head): K codes, V codes with the 16-byte pieces of slot r's row at piece c ^ (r mod 8), then
    the K and V scales) comes apart into codes in dim order and the scales."""
    from dynamic_block_sparse_gb300 import binding as B
    P, H, p = 3, 2, 16
    rng = np.random.default_rng(5)
    kc = rng.integers(0, 256, size=(P, H, p, 128), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(P, H, p, 128), dtype=np.uint8)
    ks = rng.random((P, H, p), dtype=np.float32)
    vs = rng.random((P, H, p), dtype=np.float32)
    buf = bytearray(P * H * 264 * p)
    for b in range(P):
        for h in range(H):
            base = (b * H + h) * 264 * p
            for r in range(p):
                for c in range(8):
                    at = 16 * (c ^ (r % 8))
                    buf[base + r * 128 + at: base + r * 128 + at + 16] = \
                        kc[b, h, r, 16 * c:16 * c + 16].tobytes()
                    vbase = base + 128 * p
                    buf[vbase + r * 128 + at: vbase + r * 128 + at + 16] = \
                        vc[b, h, r, 16 * c:16 * c + 16].tobytes()
            buf[base + 256 * p: base + 260 * p] = ks[b, h].tobytes()
            buf[base + 260 * p: base + 264 * p] = vs[b, h].tobytes()
    t = torch.frombuffer(buf, dtype=torch.uint8)
    k8, v8, ks8, vs8 = B.kv8_unpack(t, P, H, p)
    np.testing.assert_array_equal(k8.numpy(), kc)
    np.testing.assert_array_equal(v8.numpy(), vc)
    np.testing.assert_array_equal(ks8.numpy(), ks)
    np.testing.assert_array_equal(vs8.numpy(), vs)


def test_kv4_unpack_reads_the_documented_layout():
    """A KV4 buffer written byte by byte from the layout the header documents (per (page, KV
    head): K code rows, V code rows with slot r's 64-byte row at row r ^ ((r >> 1) & 1), then the
    K and V scales) comes apart into rows in token order and the scales."""
    from dynamic_block_sparse_gb300 import binding as B
    P, H, p = 3, 2, 16
    rng = np.random.default_rng(6)
    kc = rng.integers(0, 256, size=(P, H, p, 64), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(P, H, p, 64), dtype=np.uint8)
    ks = rng.random((P, H, p), dtype=np.float32)
    vs = rng.random((P, H, p), dtype=np.float32)
    buf = bytearray(P * H * 136 * p)
    for b in range(P):
        for h in range(H):
            base = (b * H + h) * 136 * p
            for r in range(p):
                at = 64 * (r ^ ((r >> 1) & 1))
                buf[base + at: base + at + 64] = kc[b, h, r].tobytes()
                buf[base + 64 * p + at: base + 64 * p + at + 64] = vc[b, h, r].tobytes()
            buf[base + 128 * p: base + 132 * p] = ks[b, h].tobytes()
            buf[base + 132 * p: base + 136 * p] = vs[b, h].tobytes()
    t = torch.frombuffer(buf, dtype=torch.uint8)
    k4, v4, ks4, vs4 = B.kv4_unpack(t, P, H, p)
    np.testing.assert_array_equal(k4.numpy(), kc)
    np.testing.assert_array_equal(v4.numpy(), vc)
    np.testing.assert_array_equal(ks4.numpy(), ks)
    np.testing.assert_array_equal(vs4.numpy(), vs)


def test_bench_rows_only_rejects_unknown_workload():
    """``bench.py --rows-only`` accepts the four row workloads and refuses anything else before it
    touches a GPU."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.parse_args(["--rows-only", "llama3_8b_layer"]).rows_only == "llama3_8b_layer"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--rows-only", "prr_512k"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "no rows for prr_512k" in r.stderr


def test_bench_reference_arm_prints_the_contract_line():
    """``bench.py --impl reference`` times the oracle on the host cores and prints one JSON line
    with the GPU arm's metric, unit and workload, its own cpu_baseline and an e2e equal to its
    value; under a launcher's rank other than 0 it exits 0 without output."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["config"]["workload"].startswith("prr_512k:")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r1 = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    assert r1.returncode == 0 and r1.stdout.strip() == ""


def test_stream_k_cut_geometry():
    """The persistent attention's stream-K bookkeeping, restated: CTA c of n holds the slots
    [c T / n, (c + 1) T / n) of T, and slot x belongs to CTA ((x + 1) n - 1) / T.  A row (unit) is
    cut exactly when it reaches outside the CTA's own range, and the record a cut row leaves in CTA
    c sits in slot 0 unless c is the row's first CTA and starts before the row: there the row is
    c's last unit of several, slot 1.  Checked against the division-based definitions."""
    r = np.random.default_rng(17)
    for _ in range(300):
        rows = int(r.integers(1, 40))
        stride = int(r.integers(1, 300))
        T = rows * stride
        n = int(min(r.integers(1, 153), T))
        start = lambda c: c * T // n
        owner = lambda x: ((x + 1) * n - 1) // T
        for c in range(n):
            beg, end = start(c), start(c + 1)
            assert owner(beg) == c and owner(end - 1) == c
            units = list(range(beg // stride, (end - 1) // stride + 1))
            for u, row in enumerate(units):
                rs = row * stride
                cut_by_owner = owner(rs) != owner(rs + stride - 1)
                cut_by_range = rs < beg or rs + stride > end
                assert cut_by_owner == cut_by_range
                if not cut_by_range:
                    continue
                writer_slot = 0 if u == 0 else 1       # what CTA c writes
                c_first = owner(rs)
                reader_slot = 1 if (c == c_first and start(c_first) < rs) else 0
                assert reader_slot == writer_slot
