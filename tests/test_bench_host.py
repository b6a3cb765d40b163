"""Host logic of bench.py on CPU: byte accounting, the reference arm, and the
N > 1 rank combination over a 2-process gloo group."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_prefill():
    """Compulsory bytes per kernel at B=16384, n=4, C=7168 (X read once, outputs written once)."""
    a = bench.algorithmic_bytes(16384, 4, 7168)
    assert a["gemm_rms"] == 942_538_752
    assert a["coeffs"] == 3_211_360
    assert a["pre_apply"] == 1_174_667_264
    assert a["post_res_apply"] == 2_115_239_936
    assert sum(a.values()) == 4_235_657_312


def test_kernel_bytes_prefill():
    """Steps 1-3 in one kernel: the GEMM's bytes and the coefficients' bytes, less
    the read-back of Y and r that no longer happens."""
    k = bench.kernel_bytes(16384, 4, 7168)
    assert set(k) == set(bench.KERNELS)
    assert k["gemm_rms"] == 942_538_752 + 3_211_360 - (4 * 16384 * 24 + 4 * 16384)
    assert k["pre_apply"] == 1_174_667_264
    assert k["post_res_apply"] == 2_115_239_936


def test_kernel_bytes_precision_variants():
    """The same accounting for the fp8 chain (every activation and weight value one
    byte) and the fp32-weight chain (φ as 2N bf16 rows, F_out fp32), written out."""
    B, n, C = 16384, 4, 7168
    K, N = n * C, n * n + 2 * n
    yr = 4 * B * N + 4 * B                   # Y and r, fp32
    coef = yr + 4 * N + 4 * B * (2 * n + n * n)  # Y, r, b read; H written
    hpre, hres_post = 4 * B * n, 4 * B * n * n + 4 * B * n
    e = bench.kernel_bytes(B, n, C, "e4m3")
    assert e["gemm_rms"] == B * K + N * K + yr + coef - yr == 473_661_536
    assert e["pre_apply"] == B * K + hpre + B * C == 587_464_704
    assert e["post_res_apply"] == 2 * B * K + B * C + hres_post == 1_058_275_328
    f = bench.kernel_bytes(B, n, C, "f32w")
    assert f["gemm_rms"] == 2 * B * K + 2 * (2 * N) * K + coef == 945_487_968
    assert f["pre_apply"] == 2 * B * K + hpre + 2 * B * C == 1_174_667_264
    assert f["post_res_apply"] == 4 * B * K + 4 * B * C + hres_post == 2_350_120_960


def test_tokens_per_second_is_whole_job():
    assert bench.tokens_per_second(16384, 4, 10, 1000.0) == 16384 * 4 * 10
    assert bench.max_over_ranks(3.5) == 3.5


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 150.0][rank]  # rank 1 is the slower one
    worst = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    q.put((rank, worst, bench.tokens_per_second(1000, world, 5, worst)))
    dist.barrier()
    dist.destroy_process_group()


def test_rank_combination_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [150.0, 150.0]
    assert got[0][2] == pytest.approx(1000 * 2 * 5 / 0.150)


def test_reference_arm_on_cpu():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--ref-tokens", "4"],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)  # split over every host core
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         env=env, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == ""


def test_oracle_on_all_cores_covers_every_token_once():
    """The all-core CPU baseline runs the same oracle over disjoint token ranges: its
    outputs, gathered, equal one single-threaded call over the whole range."""
    import numpy as np

    import bench
    import oracle
    import synth

    wl = synth.WORKLOADS["tiny"].with_(B=70)
    inp = synth.make_inputs(wl, 0)
    pool = bench.OracleOnAllCores(wl, inp, workers=3, chunk=16)
    got = {}
    pool._part = lambda lo, hi: got.__setitem__((lo, hi), oracle.forward(
        inp["X"][lo:hi], pool.phi, inp["F_out"][lo:hi], wl.n, wl.C, wl.alpha_pre,
        wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters))
    pool.run(0, wl.B)
    pool.close()
    assert sorted(got) == [(a, min(a + 16, 70)) for a in range(0, 70, 16)]
    whole = oracle.forward(inp["X"], pool.phi, inp["F_out"], wl.n, wl.C, wl.alpha_pre,
                           wl.alpha_post, wl.alpha_res, inp["bias"], wl.iters)
    for k in ("Y", "H_res", "X_next"):
        parts = np.concatenate([got[key][k] for key in sorted(got)])
        assert np.array_equal(parts, whole[k])


def test_stored_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed counters only while the kernel's
    source and the shared headers are those the counters were taken from: a
    change to either makes it null."""
    csrc = tmp_path / "gemm_rms_sinkhorn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "apply.cu").write_text("kernel v1\n")
    (csrc / "gemm_rms.cu").write_text("gemm v1\n")
    (csrc / "ptx.cuh").write_text("header v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest("post_res_apply")
    assert digest == bench.source_digest("pre_apply")  # same .cu file
    assert digest != bench.source_digest("gemm_rms")
    entry = {"bytes_per_launch": 123, "source_sha256_16": digest, "workload": "w"}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps({"post_res_apply": entry}))
    assert bench.stored_traffic("post_res_apply") == 123
    assert bench.stored_traffic("gemm_rms") is None  # no entry
    (csrc / "ptx.cuh").write_text("header v2\n")  # a shared header changed
    assert bench.stored_traffic("post_res_apply") is None
    (csrc / "ptx.cuh").write_text("header v1\n")
    (csrc / "apply.cu").write_text("kernel v2\n")  # the kernel's own file changed
    assert bench.stored_traffic("post_res_apply") is None


def test_committed_traffic_entries_are_well_formed():
    """Every committed entry names a timed kernel, a positive byte count and a
    16-hex-digit digest."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    for k in bench.KERNELS:
        ent = d[k]
        assert int(ent["bytes_per_launch"]) > 0
        assert len(ent["source_sha256_16"]) == 16
        int(ent["source_sha256_16"], 16)
