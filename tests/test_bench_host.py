"""Host logic of bench.py (no GPU): the kernel identity taken from a call
record, the waves of the step graph, the DRAM traffic taken
from a committed profile, the FP32 peak, the replicated (N > 1) timing
over two gloo ranks, the headline line and the reference arm's line."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gemms_linear_layers_gb300 import workloads  # noqa: E402


def test_kernel_key():
    k = bench.kernel_key
    assert k("fwd ffma nt M=2048 N=2304 K=2304 splits=1 ok") == "ffma nt"
    assert k("dgrad ffma nn M=2048 N=576 K=49152 splits=3 ok") == "ffma nn +reduce"
    assert k("fwd tc nt M=2048 N=576 K=576 batch=1 bn=64 splits=1 raster=n table=hit ok") == "tc nt bn=64"
    assert k("dgrad tc nn M=2048 N=576 K=49152 batch=1 bn=192 deep splits=3 raster=n table=hit ok") == \
        "tc nn bn=192 deep +reduce"
    assert k("wgrad tc tn M=2304 N=2304 K=2048 batch=1 bn=256 sk grid=152 raster=n table=hit ok") == "tc tn bn=256 sk"
    assert k("wgrad tc tn M=2304 N=2304 K=2048 batch=1 bn=256 splits=1 tail=10x4 raster=n table=hit ok") == \
        "tc tn bn=256 +tail"
    assert k("fwd tc nt M=2048 N=49152 K=576 batch=1 bn=256 pair splits=1 raster=m table=hit ok") == \
        "tc nt bn=256 pair"
    assert k("dgrad tc nn M=2048 N=576 K=49152 batch=1 bn=192 pair splits=3 raster=n table=hit ok") == \
        "tc nn bn=192 pair +reduce"
    assert k("fwd tc nt M=2048 N=576 K=1536 batch=1 bn=192 cs splits=1 cluster=3 raster=m table=hit ok") == \
        "tc nt bn=192 cs"
    assert k("wgrad simt tn M=200 N=300 K=520 batch=1 ok") == "simt tn"
    assert k("fwd tc3 nt M=2048 N=2304 K=13824 batch=1 bn=256 pair splits=1 raster=m table=miss ok") == \
        "tc3 nt bn=256 pair"


def _products():
    prods = []
    for dt in workloads.DECODER_135M["dtypes"]:
        for layer, d_in, d_out in workloads.LAYERS_135M:
            for op in ("fwd", "dgrad", "wgrad"):
                p = bench.Product(layer, op, dt, 2048, d_in, d_out)
                p.kernel = "tc nt bn=64"
                prods.append(p)
    return prods


def test_step_waves_cover_every_product_once_in_training_order():
    prods = _products()
    waves = bench.step_waves(prods)
    flat = [p for w in waves for p in w]
    assert sorted(map(id, flat)) == sorted(map(id, prods))
    names = [[p.name for p in w] for w in waves]
    assert names[0] == ["q.fwd.T2048.bfloat16", "k.fwd.T2048.bfloat16", "v.fwd.T2048.bfloat16"]
    assert names[5] == ["head.dgrad.T2048.bfloat16", "head.wgrad.T2048.bfloat16"]
    # a wave never mixes dtypes, and forward products come before backward ones per dtype
    for w in waves:
        assert len({p.dtype for p in w}) == 1
    order = [(p.dtype, p.op) for w in waves for p in w]
    bf = [op for dt, op in order if dt == torch.bfloat16]
    assert bf.index("dgrad") > max(i for i, op in enumerate(bf) if op == "fwd")


def test_step_waves_of_the_2b_set_keep_token_counts_apart():
    """The headline step: 7 layers x 3 products x 3 token counts x 2 dtypes,
    every wave inside one (dtype, token count) set, forwards before
    backwards within each set."""
    prods = []
    cfg = workloads.DECODER_2B
    for dt in cfg["dtypes"]:
        for T in cfg["T"]:
            for layer, d_in, d_out in cfg["layers"]:
                for op in ("fwd", "dgrad", "wgrad"):
                    prods.append(bench.Product(layer, op, dt, T, d_in, d_out))
    assert len(prods) == 126
    assert abs(sum(p.flops for p in prods) / 1e12 - 5.2510) < 1e-3
    waves = bench.step_waves(prods)
    flat = [p for w in waves for p in w]
    assert sorted(map(id, flat)) == sorted(map(id, prods))
    for w in waves:
        assert len({(p.dtype, p.T) for p in w}) == 1
    assert [p.name for p in waves[0]] == ["q.fwd.T1024.bfloat16", "k.fwd.T1024.bfloat16", "v.fwd.T1024.bfloat16"]
    assert [p.name for p in waves[4]] == ["down.dgrad.T1024.bfloat16", "down.wgrad.T1024.bfloat16"]
    p = prods[0]
    p.kernel = "tc nt bn=256 pair"
    assert p.launch_class == "tc nt bn=256 pair @ 1024x2304x2304"


def test_graph_waves_run_stream_k_alone():
    """The step graph: each wave's products side by side, except stream-K
    launches, which follow their wave one by one; serial: one product per
    wave in training order."""
    prods = []
    for T in (1024, 4096):
        for layer, d_in, d_out in workloads.DECODER_2B["layers"]:
            for op in ("fwd", "dgrad", "wgrad"):
                p = bench.Product(layer, op, torch.bfloat16, T, d_in, d_out)
                p.kernel = "tc tn bn=256 pair +tail" if op == "wgrad" else "tc nt bn=256 pair"
                prods.append(p)
    prods[-1].kernel = "tc tn bn=256 pair sk"  # down.wgrad.T4096: stream-K
    waves = bench.graph_waves(prods)
    flat = [p for w in waves for p in w]
    assert sorted(map(id, flat)) == sorted(map(id, prods))
    names = [[p.name for p in w] for w in waves]
    i = names.index(["down.dgrad.T4096.bfloat16"])
    assert names[i + 1] == ["down.wgrad.T4096.bfloat16"]
    assert ["q.dgrad.T4096.bfloat16", "q.wgrad.T4096.bfloat16", "k.dgrad.T4096.bfloat16", "k.wgrad.T4096.bfloat16",
            "v.dgrad.T4096.bfloat16", "v.wgrad.T4096.bfloat16"] in names
    assert ["q.fwd.T1024.bfloat16", "k.fwd.T1024.bfloat16", "v.fwd.T1024.bfloat16"] in names
    serial = bench.graph_waves(prods, concurrent=False)
    assert all(len(w) == 1 for w in serial) and len(serial) == len(prods)
    assert [w[0] for w in serial] == [p for w in bench.step_waves(prods) for p in w]


def test_launches_and_classes():
    assert bench.launches_of("fwd tc nt M=4096 N=5760 K=2304 batch=1 bn=256 pair splits=1 raster=m table=hit ok") == 1
    assert bench.launches_of("dgrad tc nn M=2048 N=576 K=49152 batch=1 bn=192 pair splits=3 raster=n ok") == 2
    assert bench.launches_of("wgrad tc tn M=2304 N=2304 K=2048 batch=1 bn=256 pair splits=1 tail=5x4 ok") == 2
    prods = [bench.Product("q", "fwd", torch.bfloat16, 2048, 2304, 2304),
             bench.Product("k", "fwd", torch.bfloat16, 2048, 2304, 2304),
             bench.Product("gate", "fwd", torch.bfloat16, 2048, 2304, 5760)]
    for p in prods:
        p.kernel = "tc nt bn=256 pair"
    cl = bench.by_launch_class(prods, {prods[0].name: 1.0, prods[1].name: 2.0, prods[2].name: 2.5})
    k = "tc nt bn=256 pair @ 2048x2304x2304"
    assert cl[k]["n"] == 2 and cl[k]["ms"] == 3.0 and cl[k]["flops"] == 2 * prods[0].flops
    assert max(cl.items(), key=lambda kv: kv[1]["ms"])[0] == k


def test_bars_from_rows():
    rows = [{"set": "2B", "T": 1024, "op": "fwd", "frac_cold": 0.4},
            {"set": "2B", "T": 2048, "op": "fwd", "frac_cold": 0.8},
            {"set": "2B", "T": 4096, "op": "wgrad", "frac_cold": 0.75, "wgrad_over_fwd": 0.9},
            {"set": "2B", "T": 4096, "op": "wgrad_acc", "frac_cold": 0.6},
            {"set": "LoRA", "op": "down", "frac_of_hbm": 0.5}, {"set": "LoRA", "op": "up_add", "frac_of_hbm": 0.3}]
    assert bench.bars_of(rows) == {"min_tensor_frac_T2048_4096": 0.75, "min_wgrad_over_fwd": 0.9,
                                   "min_lora_hbm_frac": 0.5}


def test_profiled_traffic_needs_matching_key_and_sources(tmp_path):
    """The roofline's DRAM traffic comes from a committed ncu summary only if
    it names the dominant kernel identity and was taken from the current
    kernel sources."""
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "gemm_tc.cuh").write_text("kernel v1\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = bench.kernel_sources_digest(str(csrc))
    (prof / "k.md").write_text("# capture\n\n- bench_kernel_key: `tc nn bn=192 pair +reduce`\n"
                               f"- traffic_bytes_per_launch: `275000000`\n- kernel_sources_sha1: `{digest}`\n")
    assert bench.profiled_traffic("tc nn bn=192 pair +reduce", str(prof), digest) == 275000000
    assert bench.profiled_traffic("tc nt bn=256 pair", str(prof), digest) is None
    (csrc / "attn_tc.cu").write_text("another unit\n")  # a unit with no kernel of the step
    assert bench.kernel_sources_digest(str(csrc)) == digest
    (csrc / "gemm_tc.cuh").write_text("kernel v2\n")  # the kernel changed since the capture
    assert bench.profiled_traffic("tc nn bn=192 pair +reduce", str(prof), bench.kernel_sources_digest(str(csrc))) is None


def test_fp32_peak_from_units_and_clock():
    """152 SMs x 128 FP32 FMA units x 2 flop x 2,070 MHz."""
    assert abs(bench.fp32_peak_tflops(152, 2070.0) - 80.5478) < 1e-3


def _two_rank_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1.0 + 1.5 r ms: every rank must see the slowest one's time
        t = bench.max_over_ranks(1.0 + 1.5 * rank, "cpu")
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(repr(t))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_time_is_the_slowest_rank_over_gloo(tmp_path):
    """The N > 1 path of the benchmark, as two gloo ranks on the CPU: the
    timed region is the maximum over ranks and the job's throughput counts
    every replica's work over that time."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_two_rank_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert float((tmp_path / f"r{r}.txt").read_text()) == 2.5
    assert bench.max_over_ranks(3.0, "cpu") == 3.0  # no process group: the rank's own time
    # 2 replicas x 10 steps x 1e12 flop in 4 s
    assert abs(bench.job_tflops(2, 1e12, 10, 4000.0) - 5.0) < 1e-12


def test_headline_line_stays_compact():
    """The last stdout line carries every key the contract asks for and stays
    under 2 KB even with the longest strings the bench can put in it."""
    import json
    roofline = {"bound": "tensor", "achieved": 1295.7, "peak": 1908.0, "unit": "TFLOP/s", "frac": 0.6791,
                "traffic": 48533248, "kernel": "tc tn bn=256 pair +tail @ 2304x2304x4096", "launches_per_step": 8,
                "gflop_per_launch": 43.487, "peak_source": "measured bf16 burst (fp16 same nominal rate)",
                "ms_per_launch": 0.03366, "share_of_step": 0.074}
    workload = bench.STEP_SETS["2b"][1]
    for mode in (bench.MODE_CONCURRENT, bench.MODE_SERIAL, bench.MODE_PER_PRODUCT):
        line = bench.headline(1437.53, 3.6528, 1, 20, 5, workload, [1024, 2048, 4096], 126,
                              "gemms_linear_layers_gb300/tables/gb300.txt", 5.251e12, 1.954e9, mode, roofline, 4040,
                              {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 4})
        line["e2e"] = {"value": 402.94, "unit": "TFLOP/s", "h2d_bytes_per_step": 1954676736,
                       "d2h_bytes_per_step": 1954676736, "ms_per_step": 13.032}
        line["cpu_baseline"] = {"value": 0.006108, "unit": "TFLOP/s", "cores": 16, "kind": "oracle",
                                "sample": "first 32 output row(s) of each of the 126 products (32.43 GMAC), fp64 "
                                          "naive loops, 10.6 s"}
        line["bars"] = {"min_tensor_frac_T2048_4096": 0.519, "min_wgrad_over_fwd": 0.752, "min_lora_hbm_frac": 0.304}
        text = json.dumps(line)
        assert len(text) < 2000, len(text)
        for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                  "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
            assert k in line, k


def test_reference_arm_line(monkeypatch, capsys):
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys, the arm's own cpu_baseline and an
    e2e of the same value without host-device traffic; the oracle's sample
    is cut short here (135M-class set) to keep the test quick."""
    import argparse
    import json
    orig = bench.oracle_sample
    monkeypatch.setattr(bench, "oracle_sample", lambda target_s, cfg=None: orig(0.2, cfg))
    bench.reference_arm(argparse.Namespace(set="135m", steps=1, warmup=0, gpus=1))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    for k in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
              "dtype", "data", "config"):
        assert k in line, k
