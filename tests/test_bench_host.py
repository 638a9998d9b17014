"""bench.py on the host: the reference arm (float64 oracle on CPU), its launch under
torchrun with two ranks, and the max-over-ranks reduction with a 2-rank gloo group."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WL = "causal_mha_S4096_h8_d64_c4"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--cpu-seconds", "1", "--workload", WL], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    j = lines[0]
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "TFLOP/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]
    assert j["config"]["workload"] == WL and j["higher_is_better"] is True


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "1", "--workload", WL],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 5.0 - rank]          # rank 1 slower in the step, faster end to end
    got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 5.0]


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_value(1e12, 1, 1000.0)
    assert abs(one - 1.0) < 1e-12
    assert abs(bench.whole_job_value(1e12, 4, 1000.0) - 4.0) < 1e-12


def test_code_fingerprint_ignores_comments_only(tmp_path, monkeypatch):
    """The traffic record is keyed by a fingerprint of the attention kernel's code (its source
    and the headers it includes): editing a comment keeps it, editing code in any of the files
    changes it."""
    sys.path.insert(0, ROOT)
    import bench
    srcs = [open(p, encoding="utf-8").read() for p in bench.KERNEL_SRCS]

    def fingerprint(texts, tag):
        paths = []
        for i, t in enumerate(texts):
            q = tmp_path / f"{tag}_{i}"
            q.write_text(t, encoding="utf-8")
            paths.append(str(q))
        monkeypatch.setattr(bench, "KERNEL_SRCS", tuple(paths))
        return bench.src_hash()

    h0 = fingerprint(srcs, "base")
    assert h0 == fingerprint(srcs, "again")
    commented = ["// a new comment line\n" + srcs[0].replace("namespace ra {", "namespace ra {  /* note */", 1)]
    commented += [srcs[1] + "\n// trailing note\n", srcs[2]]
    assert fingerprint(commented, "commented") == h0
    changed = [srcs[0].replace("constexpr int kThreads = 352;", "constexpr int kThreads = 384;", 1)] + srcs[1:]
    assert changed[0] != srcs[0] and fingerprint(changed, "kernel") != h0
    marker = "__device__ __forceinline__ bool mbar_wait_noabort("
    assert marker in srcs[1]
    header = [srcs[0], srcs[1].replace(marker, "__device__ __noinline__ bool mbar_wait_noabort(", 1), srcs[2]]
    assert fingerprint(header, "header") != h0


def _row_parity_case():
    """A small causal GQA case whose 'device result' is the oracle's own, in host float32."""
    from types import SimpleNamespace
    from oracle.attention import full_attention
    g = torch.Generator().manual_seed(41)
    q = torch.randn((4, 48, 16), generator=g).to(torch.bfloat16)
    k = torch.randn((2, 48, 16), generator=g).to(torch.bfloat16)
    v = torch.randn((2, 48, 16), generator=g).to(torch.bfloat16)
    o, l = full_attention(*(x.double().numpy() for x in (q, k, v)), True)
    w = SimpleNamespace(bhq=4, seq=48, causal=1, d=16)
    return w, (q, k, v), torch.from_numpy(o).float(), torch.from_numpy(l).float()


def test_bench_row_parity_reports_the_sampled_rows():
    """The bench line's `parity` entry: the cpu_baseline leg's oracle rows against a result in
    host memory -- exact agreement passes, a planted error or a NaN row fails, and a failure
    inside the comparison is recorded instead of raised."""
    sys.path.insert(0, ROOT)
    import bench
    w, qkv, out_h, lse_h = _row_parity_case()

    check = bench.RowParity(out_h, lse_h, "host copy")
    units = bench.cpu_oracle_units(w, qkv, 0.0, min_units=2, check=check)
    s = check.summary()
    assert len(units) == 2 and s["rows"] == 2 * 4 * 48   # each unit samples every row here
    assert s["within_tolerance"] and s["error"] is None and s["nonfinite_rows"] == 0
    assert s["max_abs_err_out"] < 1e-6 and s["max_abs_err_lse"] < 1e-5

    bad = out_h.clone()
    bad[3, 47, 5] += 0.05
    check = bench.RowParity(bad, lse_h, "host copy")
    bench.cpu_oracle_units(w, qkv, 0.0, check=check)
    s = check.summary()
    assert not s["within_tolerance"] and abs(s["max_abs_err_out"] - 0.05) < 1e-3

    nan = lse_h.clone()
    nan[1, 0] = float("nan")
    check = bench.RowParity(out_h, nan, "host copy")
    bench.cpu_oracle_units(w, qkv, 0.0, check=check)
    s = check.summary()
    assert s["nonfinite_rows"] == 1 and not s["within_tolerance"]

    check = bench.RowParity(out_h[:, :8], lse_h, "host copy")   # too short: indexing fails
    bench.cpu_oracle_units(w, qkv, 0.0, check=check)
    s = check.summary()
    assert s["error"] is not None and not s["within_tolerance"]
