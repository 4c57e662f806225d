"""Benchmark of the IQ hot path on B300.

Workload (the pages' encode-speed configuration): one 5632 x 2048 bf16 weight (Student-t nu=4 x
0.02), importance from 4096 x 2048 bf16 activations with log-normal column scales, seeded synthetic
codebooks.  One step = the whole hot path over that batch:
  imatrix accumulation (1024-row chunks) -> importance weights -> for each of the five formats:
  searched encode with the every-choice error table (anchor fused) + fixed-choice encode (choice 7
  everywhere) + decode of the searched payload (fp32).
value = 5 * 5632 * 2048 weight elements / step time (M elem/s; each element goes through the full
path once per format).  Per-kernel CUDA-event times give per-format encode M elem/s, decode and
imatrix GB/s and the roofline of the dominant kernel.  Besides the step, the line reports the
routed-MoE imatrix (4096 x 17408, 128 experts), the HBM-bound large-layer decode, the MoE expert
encode (128 x [1536, 2048]), the large-layer encode with every-choice tables ([17408, 5120] and
[5120, 17408]) and the local-Hessian choice search.

--impl reference times the plain C oracle (the CPU definition of the same path) on a bounded row
sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "IQ encode M elem/s per format on 5632x2048 (+% FP32 roofline); imatrix/decode GB/s"
R, C = 5632, 2048
T_ACT = 4096
FORMATS = ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M")
ENTRIES = {"IQ2_XXS": 256, "IQ2_XS": 512, "IQ2_S": 1024, "IQ1_S": 2048, "IQ1_M": 2048}
BPW = {"IQ2_XXS": 2.0625, "IQ2_XS": 2.3125, "IQ2_S": 2.5625, "IQ1_S": 1.5625, "IQ1_M": 1.75}
CONFIG = {"workload": "encode 5632x2048 bf16 weight in IQ2_XXS/IQ2_XS/IQ2_S/IQ1_S/IQ1_M (searched + every-choice "
                      "table, fixed choice 7, decode) with importance from a 4096x2048 bf16 imatrix pass",
          "rows": R, "cols": C, "activation_rows": T_ACT, "rows_per_chunk": 1024,
          "l2": "flushed before every timed step (512 MiB write); inputs 23 MiB + 16 MiB < L2",
          "timing": "one CUDA graph of the whole step per timed step, CUDA events on the launching stream"}


MOE_T, MOE_C, MOE_E, MOE_K = 4096, 17408, 128, 8
DEC_R, DEC_C = 17408, 5120
EXP_E, EXP_R, EXP_C = 128, 1536, 2048          # MoE expert encode: 128 x gate/up [1536, 2048]
LARGE_SHAPES = ((17408, 5120), (5120, 17408))  # large-layer encode with the every-choice table
REF_CONFIG = {"workload": CONFIG["workload"], "rows": R, "cols": C, "activation_rows": T_ACT,
              "rows_per_chunk": 1024,
              "timing": "host wall clock over whole steps of the plain C oracle (fp64 direct-form search, "
                        "OpenMP over blocks) on this host's cores; each step encodes a row sample"}

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the searched encode
# kernel on this workload, from ncu captures of that launch, and the SHA-256 of the encoder
# sources they were taken on: the figure is reported only while the sources are unchanged.
PROFILED_ENCODE_TRAFFIC = {"IQ2_XXS": 23197440, "IQ1_S": 23277568, "IQ1_M": 23298048}
PROFILED_ENCODE_SHA256 = "68101d4cbefd7424c847e1693af7f00d64b204938e3087f0e184c7e799a6ffce"
ENCODE_SOURCES = ("ggml_iq_codebook_accumulate_b300/csrc/iq_encode.cu", "ggml_iq_codebook_accumulate_b300/csrc/iq_common.cuh")


def measured_peaks():
    """HBM copy bandwidth (GB/s) measured on this GPU pool, else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


def encode_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for f in ENCODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def flops_per_element(fmt):
    """Algorithmic FP32 work of the searched encode per weight element: per codebook entry and
    8-value vector, IQ2 16 FMA for (A, B) + 16 choices x (FMA + min) = 80 flops; IQ1 24 FMA +
    4 shifted-form FMA + 16 x (FMA + min) = 104 flops (FMA = 2, min = 1)."""
    return (10 if fmt.startswith("IQ2") else 13) * ENTRIES[fmt]


def cuda_core_flops_per_element(fmt):
    """The part of the cost model that still runs on the FP32 lanes once the per-entry dot
    products run on the tensor cores: per entry and vector, 16 choices x (FMA + min) = 48 flops for
    IQ2; IQ1 adds 5 FMAs for the shifted sums: 58 flops."""
    return (6.0 if fmt.startswith("IQ2") else 7.25) * ENTRIES[fmt]


def fp32_peak_tflops(sms, mhz):
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def inputs():
    from ggml_iq_codebook_accumulate_b300 import synth
    Wst, Wv = synth.as_dtype(synth.weight_t4(R, C, seed=1), "bf16")
    Xst, Xv = synth.as_dtype(synth.activations(T_ACT, C, seed=1), "bf16")
    grids = {f: synth.grid(f) for f in FORMATS}
    return Wst, Wv, Xst, Xv, grids


# ----------------------------------------------------------------------------------------------
def run_reference(args):
    """The oracle (plain C, fp64 direct-form search, OpenMP over blocks) on a bounded row sample."""
    import oracle
    oracle.build()
    Wst, Wv, Xst, Xv, grids = inputs()
    rows = int(os.environ.get("IQ_REF_ROWS", "128"))
    ids = np.zeros((T_ACT, 1), np.int32)

    def step():
        s2, cn, _ = oracle.imatrix_accumulate(Xv, ids, 1)
        w = oracle.imatrix_weights(s2, cn)[0]
        for f in FORMATS:
            p, _ = oracle.encode(f, Wv[:rows], grids[f], importance=w)
            ch = np.full((rows * C // 256, oracle.format_info(f)["groups"]), 7, np.uint8)
            oracle.encode(f, Wv[:rows], grids[f], importance=w, choices=ch)
            oracle.decode(f, p, rows, C, grids[f])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = 5 * rows * C / dt / 1e6
    cores = os.cpu_count()
    sample = (f"{rows} of {R} rows per format (searched + fixed-choice encode, decode) plus the full "
              f"{T_ACT}x{C} imatrix pass, per step")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "M elem/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(REF_CONFIG, rows_sampled=rows),
            "cpu_baseline": {"value": round(value, 4), "unit": "M elem/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "M elem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline_sample(Wv, Xv, grids, budget_rows=768, single_rows=48):
    """The oracle on this host: all cores (OpenMP over blocks) on ``budget_rows`` rows per format,
    and one thread on ``single_rows`` rows, each with the full imatrix pass (single-threaded in the
    oracle) once."""
    import oracle
    oracle.build()
    ids = np.zeros((T_ACT, 1), np.int32)

    def run(rows, threads):
        t0 = time.perf_counter()
        s2, cn, _ = oracle.imatrix_accumulate(Xv, ids, 1)
        w = oracle.imatrix_weights(s2, cn)[0]
        for f in FORMATS:
            p, _ = oracle.encode(f, Wv[:rows], grids[f], importance=w, threads=threads)
            ch = np.full((rows * C // 256, oracle.format_info(f)["groups"]), 7, np.uint8)
            oracle.encode(f, Wv[:rows], grids[f], importance=w, choices=ch, threads=threads)
            oracle.decode(f, p, rows, C, grids[f])
        return time.perf_counter() - t0

    dt = run(budget_rows, 0)
    dt1 = run(single_rows, 1)
    return {"value": round(5 * budget_rows * C / dt / 1e6, 4), "unit": "M elem/s", "cores": os.cpu_count(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"one step on {budget_rows} of {R} rows per format (searched + fixed encode, decode) plus the "
                      f"full {T_ACT}x{C} imatrix pass; {dt:.1f} s",
            "single_thread": {"value": round(5 * single_rows * C / dt1 / 1e6, 4), "unit": "M elem/s", "cores": 1,
                              "sample": f"one step on {single_rows} rows per format plus the imatrix pass, one "
                                        f"thread; {dt1:.1f} s"}}


# ----------------------------------------------------------------------------------------------
class Clocks:
    def __init__(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        dev = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0] or "0"
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", dev, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                       "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            self.p.wait()

    def summary(self):
        self.f.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1])); mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def run_ours(args):
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, replicas

    rank, world, local = replicas.world_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    api.lib()
    Wst, Wv, Xst, Xv, grids = inputs()

    def to_dev(store):
        return torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)

    W = to_dev(Wst)
    X = to_dev(Xst)
    G = {f: torch.from_numpy(grids[f]).to(dev) for f in FORMATS}
    ids = torch.zeros(T_ACT, 1, dtype=torch.int32, device=dev)
    s2 = torch.zeros(1, C, dtype=torch.float32, device=dev)
    cn = torch.zeros(1, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B = R * C // 256
    info = {f: api.format_info(f) for f in FORMATS}
    pay = {f: torch.empty(B, info[f]["block_bytes"], dtype=torch.uint8, device=dev) for f in FORMATS}
    pay7 = {f: torch.empty_like(pay[f]) for f in FORMATS}
    tbl = {f: torch.empty(B, info[f]["choice_groups"], info[f]["num_choices"], dtype=torch.float32, device=dev)
           for f in FORMATS}
    ch7 = {f: torch.full((B, info[f]["choice_groups"]), 7, dtype=torch.uint8, device=dev) for f in FORMATS}
    dec = torch.empty(R, C, dtype=torch.float32, device=dev)
    ws = {f: api.encode_workspace(f, R, C, dev) for f in FORMATS}
    ws_im = api.imatrix_workspace(T_ACT, C, torch.bfloat16, 1, 1, 1024, dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    wbuf = {}

    def c_imatrix():
        s2.zero_(); cn.zero_()
        api.imatrix_accumulate(X, ids, 1, 1024, s2, cn, status=st, workspace=ws_im)

    def c_weights():
        wbuf["w"] = api.imatrix_weights(s2, cn)

    def c_encode(f):
        api.encode(f, W, G[f], importance=wbuf["w"][0], status=st, payload=pay[f], table=tbl[f], every_choice=True,
                   workspace=ws[f])

    def c_fixed(f):
        api.encode(f, W, G[f], importance=wbuf["w"][0], choices=ch7[f], status=st, payload=pay7[f], workspace=ws[f])

    def c_decode(f):
        api.decode(f, pay[f], R, C, G[f], out=dec)

    parts = [("imatrix", c_imatrix), ("weights", c_weights)]
    for f in FORMATS:
        parts += [(f"encode:{f}", lambda f=f: c_encode(f)), (f"fixed:{f}", lambda f=f: c_fixed(f)),
                  (f"decode:{f}", lambda f=f: c_decode(f))]

    def step():
        for _, fn in parts:
            fn()

    if args.only:
        run_only(args, dev, dict(parts), flush, stream)
        return
    for _ in range(args.warmup):                       # eager warm-up (loads modules, sets attributes)
        step()
    torch.cuda.synchronize()
    # The step and each of its calls are captured as CUDA graphs: a replay runs exactly the
    # library's kernels of the step with no host launch gaps.
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step()
    g_part = {}
    for name, fn in parts:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g_part[name] = g
    for _ in range(2):
        g_step.replay()
    torch.cuda.synchronize()
    replicas.barrier()

    def timed(g):
        flush.fill_(1)                                 # L2 flushed before every timed replay
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        return a, b

    totals = []
    with Clocks() as clk:
        torch.cuda.synchronize()
        evs = [timed(g_step) for _ in range(args.steps)]
        torch.cuda.synchronize()
        totals = [a.elapsed_time(b) for a, b in evs]
    replicas.barrier()
    per = {n: [] for n, _ in parts}
    for _ in range(max(3, args.steps)):
        evs = {n: timed(g_part[n]) for n, _ in parts}
        torch.cuda.synchronize()
        for n, (a, b) in evs.items():
            per[n].append(a.elapsed_time(b))
    ms = replicas.max_over_ranks(float(np.mean(totals)), device=dev)
    if rank != 0:
        return
    clocks = clk.summary()
    value = replicas.job_throughput(5 * R * C, ms * 1e-3, world) / 1e6
    # per-kernel figures
    pf = {}
    for f in FORMATS:
        e_ms = float(np.mean(per[f"encode:{f}"]))
        x_ms = float(np.mean(per[f"fixed:{f}"]))
        d_ms = float(np.mean(per[f"decode:{f}"]))
        dec_bytes = R * C * (BPW[f] / 8 + 4) + ENTRIES[f] * 32
        pf[f] = {"encode_searched_Melem_s": round(R * C / (e_ms * 1e-3) / 1e6, 1),
                 "encode_fixed_Melem_s": round(R * C / (x_ms * 1e-3) / 1e6, 1),
                 "decode_GB_s": round(dec_bytes / (d_ms * 1e-3) / 1e9, 1),
                 "encode_ms": round(e_ms, 4), "fixed_ms": round(x_ms, 4), "decode_ms": round(d_ms, 4)}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    im_ms = float(np.mean(per["imatrix"]))
    im_bytes = T_ACT * C * 2 + T_ACT * 4 + 2 * C * 4
    hbm, hbm_src = measured_peaks()
    moe = measure_imatrix_moe(args, dev, flush, hbm)
    dec_large = measure_decode_large(args, dev, flush, hbm)
    lhs = measure_local_hessian(args, dev, flush)
    moe_enc = measure_moe_expert_encode(args, dev, flush)
    wb = measure_write_back(args, dev, flush, W, G, wbuf["w"][0])
    large = measure_large_layers(args, dev, flush)
    for f in FORMATS:
        # the step's 46 MB fp32 output stays in L2: this is an L2-resident rate, not an HBM one
        pf[f]["decode_note"] = "output L2-resident (46 MB < L2); the HBM-bound decode is decode_large"
        pf[f]["encode_searched_frac_fp32"] = _encode_figures(f, R * C, pf[f]["encode_ms"], sms)["frac_fp32"]
        pf[f]["encode_searched_frac_cuda_core_work"] = _encode_figures(f, R * C, pf[f]["encode_ms"], sms)["frac_cuda_core_work"]
    dom = max(FORMATS, key=lambda f: pf[f]["encode_ms"])
    dom_ms = pf[dom]["encode_ms"]
    achieved = R * C * flops_per_element(dom) / (dom_ms * 1e-3) / 1e12
    peak = fp32_peak_tflops(sms, 2032.0)
    prof_traffic = (PROFILED_ENCODE_TRAFFIC.get(dom) if encode_sources_sha256() == PROFILED_ENCODE_SHA256 else None)
    achieved_cc = R * C * cuda_core_flops_per_element(dom) / (dom_ms * 1e-3) / 1e12
    roofline = {"kernel": f"iq_encode call {dom} (prep_codebook + encode_tc_kernel + rescore_kernel; searched + "
                          "every-choice table)", "bound": "alu",
                "achieved": round(achieved, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": prof_traffic,
                "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 flops x 2032 MHz (max SM clock)",
                "flops_per_element": flops_per_element(dom),
                "frac_cuda_core_work": round(achieved_cc / peak, 4)}
    if clocks.get("sm_mhz"):
        roofline["frac_at_observed_clock"] = round(achieved / fp32_peak_tflops(sms, clocks["sm_mhz"]), 4)
    # end to end through the public API with host buffers
    e2e = measure_e2e(args, dev, Wst, Xst, grids, G, ids, info)
    # this library's kernels per step: imatrix route + csr + accumulate (+ combine when chunks run
    # in parallel), weights, and per format: codebook prep + encode + rescore (searched and fixed)
    # and decode
    im_kernels = 4 if T_ACT > 1024 and (C + 127) // 128 < 112 else 3
    launches = args.steps * (im_kernels + 1 + len(FORMATS) * (3 + 3 + 1))
    cpu = cpu_baseline_sample(Wv, Xv, grids) if world == 1 or rank == 0 else None
    line = {"metric": METRIC, "value": round(value, 2), "unit": "M elem/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": CONFIG,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
            "per_format": pf,
            "imatrix": {"ms": round(im_ms, 4), "GB_s": round(im_bytes / (im_ms * 1e-3) / 1e9, 1),
                        "frac_hbm": round(im_bytes / (im_ms * 1e-3) / 1e9 / hbm, 4)},
            "imatrix_moe": moe, "decode_large": dec_large, "local_hessian": lhs, "moe_expert_encode": moe_enc,
            "large_layer_encode": large, "write_back": wb, "hbm_peak_GB_s": hbm, "hbm_peak_source": hbm_src}
    print(json.dumps(line))


def run_only(args, dev, fns, flush, stream):
    """One part of the step on its own (the profiling runs): --warmup untimed eager calls, then
    --steps calls each timed with CUDA events after an L2 flush.  Parts: imatrix, weights,
    encode:<fmt>, fixed:<fmt>, decode:<fmt>, imatrix_moe, decode_large, local_hessian,
    moe_expert_encode, large_layer_encode."""
    import torch
    if args.only in ("imatrix_moe", "decode_large"):
        hbm, _ = measured_peaks()
        fn = measure_imatrix_moe if args.only == "imatrix_moe" else measure_decode_large
        print(json.dumps({"only": args.only, **fn(args, dev, flush, hbm)}))
        return
    if args.only == "local_hessian":
        print(json.dumps({"only": args.only, **measure_local_hessian(args, dev, flush)}))
        return
    if args.only in ("moe_expert_encode", "large_layer_encode"):
        fn = measure_moe_expert_encode if args.only == "moe_expert_encode" else measure_large_layers
        print(json.dumps({"only": args.only, **fn(args, dev, flush)}))
        return
    if args.only not in fns:
        extra = ['imatrix_moe', 'decode_large', 'local_hessian', 'moe_expert_encode', 'large_layer_encode']
        raise SystemExit(f"--only: unknown part {args.only!r}; one of {sorted(fns) + extra}")
    fns["imatrix"]()
    fns["weights"]()
    fn = fns[args.only]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.fill_(3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    print(json.dumps({"only": args.only, "steps": args.steps, "warmup": args.warmup,
                      "ms_mean": round(float(np.mean(times)), 4), "ms_min": round(float(np.min(times)), 4)}))


def measure_decode_large(args, dev, flush, hbm):
    """Decode of one large-layer weight, 17408 x 5120 (Student-t nu=4 x 0.02, bf16), from its
    searched IQ2_XXS payload to fp32.  The 356.5 MB output is about three times L2, so the kernel
    writes to HBM.  Algorithmic bytes: the payload read once, the codebook, the output written."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, synth
    store, _ = synth.as_dtype(synth.weight_t4(DEC_R, DEC_C, seed=4), "bf16")
    W = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)
    g = torch.from_numpy(synth.grid("IQ2_XXS")).to(dev)
    pay = api.encode("IQ2_XXS", W, g)
    del W
    out = torch.empty(DEC_R, DEC_C, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        api.decode("IQ2_XXS", pay, DEC_R, DEC_C, g, out=out)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        api.decode("IQ2_XXS", pay, DEC_R, DEC_C, g, out=out)
    times = []
    for _ in range(max(5, args.steps)):
        flush.fill_(4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gr.replay()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    nbytes = pay.numel() + out.numel() * 4 + g.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"IQ2_XXS payload of a {DEC_R}x{DEC_C} bf16 weight -> fp32", "ms": round(ms, 4),
            "GB_s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4), "algorithmic_bytes": int(nbytes)}


LH_R, LH_C = 4096, 2048
LH_PAGES_MS = {"IQ2_XXS": 4.8, "IQ2_S": 9.0, "IQ1_S": 5.3}   # per 256-column block of 4096 rows, GB300


def lh_inputs():
    """A 4096 x 2048 bf16 weight (Student-t nu=4 x 0.02) and the input Hessian H = X^T X / n of
    4096 correlated activations (AR(1) along the columns, coefficient 0.85, log-normal column
    scales), as its 256 x 256 diagonal blocks; importance sqrt(diag(H)) as on the pages."""
    from ggml_iq_codebook_accumulate_b300 import synth
    store, _ = synth.as_dtype(synth.weight_t4(LH_R, LH_C, seed=5), "bf16")
    rng = np.random.default_rng(5)
    Z = rng.standard_normal((4096, LH_C))
    X = np.empty_like(Z)
    X[:, 0] = Z[:, 0]
    for j in range(1, LH_C):
        X[:, j] = 0.85 * X[:, j - 1] + np.sqrt(1 - 0.85 ** 2) * Z[:, j]
    X *= np.exp(0.5 * rng.standard_normal(LH_C))[None, :]
    H = X.T @ X / X.shape[0]
    Hb = np.stack([H[256 * j:256 * (j + 1), 256 * j:256 * (j + 1)] for j in range(LH_C // 256)]).astype(np.float32)
    return store, Hb, np.sqrt(np.diag(H)).astype(np.float32)


def measure_local_hessian(args, dev, flush):
    """Every-choice encode and local-Hessian choice search of a 4096 x 2048 bf16 weight, per
    256-column block (the pages' unit: GB300, 4096 rows)."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, synth
    store, Hb, imp = lh_inputs()
    W = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)
    H = torch.from_numpy(Hb).to(dev)
    w = torch.from_numpy(imp).to(dev)
    stream = torch.cuda.current_stream(dev)
    out = {"workload": f"{LH_R}x{LH_C} bf16 weight, H from 4096 correlated activations, perc_damp 0.3"}
    for f in LH_PAGES_MS:
        g = torch.from_numpy(synth.grid(f)).to(dev)
        ws = api.encode_workspace(f, LH_R * api.format_info(f)["num_choices"], LH_C, dev)
        lws = api.local_hessian_workspace(f, LH_R, LH_C, dev)
        pay = api.encode_every_choice(f, W, g, importance=w, workspace=ws)
        ch = api.local_hessian_choices(f, W, g, pay, H, 0.3, workspace=lws)

        def t(fn):
            fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(max(3, args.steps)):
                flush.fill_(5)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            return float(np.median(ts))

        ec = t(lambda: api.encode_every_choice(f, W, g, importance=w, payloads=pay, workspace=ws))
        se = t(lambda: api.local_hessian_choices(f, W, g, pay, H, 0.3, choices=ch, workspace=lws))
        nblk = LH_C // 256
        out[f] = {"every_choice_ms": round(ec, 4), "search_ms": round(se, 4),
                  "ms_per_256col_block": round((ec + se) / nblk, 4),
                  "pages_gb300_ms_per_256col_block": LH_PAGES_MS[f]}
    return out


def measure_imatrix_moe(args, dev, flush, hbm):
    """The routed-MoE imatrix workload: 4096 tokens x 17408-wide bf16 activations (log-normal
    column scales), 128 experts, top-8 from a Zipf(1.2) router with 8 idle experts, 1,024-row
    chunks.  Algorithmic bytes: x and the ids read once, in_sum2 of the touched experts read and
    written once."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, synth
    xs, _ = synth.as_dtype(synth.activations(MOE_T, MOE_C, seed=2), "bf16")
    ids_np = synth.router(MOE_T, MOE_E, MOE_K, seed=2)
    X = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(dev)
    ids = torch.from_numpy(ids_np).to(dev)
    s2 = torch.zeros(MOE_E, MOE_C, dtype=torch.float32, device=dev)
    cn = torch.zeros(MOE_E, dtype=torch.int64, device=dev)
    ws = api.imatrix_workspace(MOE_T, MOE_C, torch.bfloat16, MOE_E, MOE_K, 1024, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        api.imatrix_accumulate(X, ids, MOE_E, 1024, s2, cn, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        api.imatrix_accumulate(X, ids, MOE_E, 1024, s2, cn, workspace=ws)
    times = []
    for _ in range(max(5, args.steps)):
        flush.fill_(2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    counts = np.bincount(ids_np.ravel(), minlength=MOE_E)
    touched = int((counts > 0).sum())
    nbytes = MOE_T * MOE_C * 2 + ids_np.nbytes + 2 * touched * MOE_C * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"{MOE_T}x{MOE_C} bf16, {MOE_E} experts, top-{MOE_K} Zipf(1.2), 1024-row chunks",
            "ms": round(ms, 4), "GB_s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
            "algorithmic_bytes": nbytes, "idle_experts": int((counts == 0).sum()),
            "tokens_per_expert_min_median_max": [int(counts.min()), int(np.median(counts)), int(counts.max())]}


def _time_call(fn, args, flush, stream, fill):
    """Median CUDA-event time (ms) of ``fn`` over max(3, steps) calls, L2 flushed before each."""
    import torch
    fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(3, args.steps)):
        flush.fill_(fill)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return float(np.median(ts))


def _encode_figures(fmt, nelem, ms, sms):
    tf = nelem * flops_per_element(fmt) / (ms * 1e-3) / 1e12
    tf_cc = nelem * cuda_core_flops_per_element(fmt) / (ms * 1e-3) / 1e12
    peak = fp32_peak_tflops(sms, 2032.0)
    return {"ms": round(ms, 4), "Melem_s": round(nelem / (ms * 1e-3) / 1e6, 1),
            "frac_fp32": round(tf / peak, 4), "frac_cuda_core_work": round(tf_cc / peak, 4)}


def measure_moe_expert_encode(args, dev, flush):
    """MoE expert encode: 128 experts x a fused gate/up weight [1536, 2048] bf16 (Student-t nu=4 x
    0.02) in one call per format (rows_per_expert 1536), each expert weighted by its own imatrix
    slice from 4096 routed tokens (top-8 of a Zipf(1.2) router with 8 idle experts, whose weight
    is 1), searched choices."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, synth
    xs, _ = synth.as_dtype(synth.activations(T_ACT, EXP_C, seed=3), "bf16")
    ids = torch.from_numpy(synth.router(T_ACT, EXP_E, 8, seed=3)).to(dev)
    X = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(dev)
    s2, cn = api.imatrix_accumulate(X, ids, EXP_E)
    w = api.imatrix_weights(s2, cn)
    del X
    store, _ = synth.as_dtype(synth.weight_t4(EXP_E * EXP_R, EXP_C, seed=3), "bf16")
    W = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nelem = EXP_E * EXP_R * EXP_C
    out = {"workload": f"{EXP_E} experts x [{EXP_R}, {EXP_C}] bf16, per-expert importance, searched"}
    for f in ("IQ2_XXS", "IQ1_M"):
        g = torch.from_numpy(synth.grid(f)).to(dev)
        ws = api.encode_workspace(f, EXP_E * EXP_R, EXP_C, dev)
        pay = api.encode(f, W, g, importance=w, rows_per_expert=EXP_R, workspace=ws)
        ms = _time_call(lambda: api.encode(f, W, g, importance=w, rows_per_expert=EXP_R, payload=pay, workspace=ws),
                        args, flush, stream, 6)
        out[f] = _encode_figures(f, nelem, ms, sms)
    return out


def measure_large_layers(args, dev, flush):
    """Large-layer encode: [17408, 5120] and [5120, 17408] bf16 weights (Student-t nu=4 x 0.02) in
    all five formats, searched, with the every-choice error table written next to the payload;
    importance from 4096 log-normal-scaled activations."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api, synth
    stream = torch.cuda.current_stream(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for (r, c) in LARGE_SHAPES:
        xs, _ = synth.as_dtype(synth.activations(T_ACT, c, seed=4), "bf16")
        X = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(dev)
        s2, cn = api.imatrix_accumulate(X, torch.zeros(T_ACT, 1, dtype=torch.int32, device=dev), 1)
        w = api.imatrix_weights(s2, cn)[0]
        del X
        store, _ = synth.as_dtype(synth.weight_t4(r, c, seed=4), "bf16")
        W = torch.from_numpy(np.ascontiguousarray(store).view(np.int16)).view(torch.bfloat16).to(dev)
        key = f"{r}x{c}"
        out[key] = {}
        for f in FORMATS:
            g = torch.from_numpy(synth.grid(f)).to(dev)
            ws = api.encode_workspace(f, r, c, dev)
            pay, tbl = api.encode(f, W, g, importance=w, every_choice=True, workspace=ws)
            ms = _time_call(lambda: api.encode(f, W, g, importance=w, payload=pay, table=tbl, every_choice=True,
                                               workspace=ws), args, flush, stream, 7)
            out[key][f] = _encode_figures(f, r * c, ms, sms)
            out[key][f]["table_MB"] = round(tbl.numel() * 4 / 1e6, 1)
            del pay, tbl, ws
        del W
        torch.cuda.empty_cache()
    return out


def measure_write_back(args, dev, flush, W0, G, w):
    """Encode with write-back of the decoded weight (one call, fused) against a separate encode and
    decode, on the step's 5632 x 2048 bf16 weight with its importance (searched choices).  W is
    restored from a copy before each timed call, outside the timed region."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api
    stream = torch.cuda.current_stream(dev)
    Wt = torch.empty_like(W0)
    out = {}
    for f in FORMATS:
        ws = api.encode_workspace(f, R, C, dev)
        pay = api.encode(f, W0, G[f], importance=w, workspace=ws)
        dec = torch.empty_like(W0)

        def fused():
            api.encode_write_back(f, Wt, G[f], importance=w, payload=pay, workspace=ws)

        def separate():
            api.encode(f, Wt, G[f], importance=w, payload=pay, workspace=ws)
            api.decode(f, pay, R, C, G[f], out=dec)

        res = {}
        for name, fn in (("fused_ms", fused), ("encode_then_decode_ms", separate)):
            ts = []
            for _ in range(max(3, args.steps) + 1):
                Wt.copy_(W0)
                flush.fill_(8)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            res[name] = round(float(np.median(ts[1:])), 4)
        out[f] = res
    return out


def measure_e2e(args, dev, Wst, Xst, grids, G, ids, info):
    """The same step through the public API with host inputs: pinned host -> device copies of the
    weight and activations, and device -> host copies of the five searched payloads and their
    every-choice error tables, all inside the timed region.  The steps are pipelined as a
    production loop would run them: each step's inputs are copied into one of two device buffers
    on their own stream while the previous step computes (the first step's copy is not
    overlapped), and each format's outputs are copied back on a second stream while the next
    format is encoded; the region ends when every stream is done."""
    import torch

    from ggml_iq_codebook_accumulate_b300 import api
    Wh = torch.from_numpy(np.ascontiguousarray(Wst).view(np.int16)).view(torch.bfloat16).pin_memory()
    Xh = torch.from_numpy(np.ascontiguousarray(Xst).view(np.int16)).view(torch.bfloat16).pin_memory()
    B = R * C // 256
    outs = {f: torch.empty(B, info[f]["block_bytes"], dtype=torch.uint8).pin_memory() for f in FORMATS}
    touts = {f: torch.empty(B, info[f]["choice_groups"], info[f]["num_choices"], dtype=torch.float32).pin_memory()
             for f in FORMATS}
    Wd = [torch.empty(R, C, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    Xd = [torch.empty(T_ACT, C, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ch7 = {f: torch.full((B, info[f]["choice_groups"]), 7, dtype=torch.uint8, device=dev) for f in FORMATS}

    compute = torch.cuda.current_stream(dev)
    copier = torch.cuda.Stream(dev)     # results back to the host
    loader = torch.cuda.Stream(dev)     # the next step's inputs to the device
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def load(k):
        with torch.cuda.stream(loader):
            if k >= 2:
                loader.wait_event(free[k % 2])        # step k - 2 is done with this buffer
            Wd[k % 2].copy_(Wh, non_blocking=True)
            Xd[k % 2].copy_(Xh, non_blocking=True)
            ready[k % 2].record(loader)

    def step(k, last):
        compute.wait_event(ready[k % 2])
        if not last:
            load(k + 1)
        W, X = Wd[k % 2], Xd[k % 2]
        s2, cn = api.imatrix_accumulate(X, ids, 1, 1024)
        w = api.imatrix_weights(s2, cn)
        for f in FORMATS:
            p, t = api.encode(f, W, G[f], importance=w[0], every_choice=True)
            copier.wait_stream(compute)               # the payload is complete
            with torch.cuda.stream(copier):
                outs[f].copy_(p, non_blocking=True)
                touts[f].copy_(t, non_blocking=True)
            p.record_stream(copier)                   # not reused before its copy is done
            t.record_stream(copier)
            api.encode(f, W, G[f], importance=w[0], choices=ch7[f])
            api.decode(f, p, R, C, G[f])
        free[k % 2].record(compute)

    def run(n):
        load(0)
        for k in range(n):
            step(k, k == n - 1)
        compute.synchronize()
        copier.synchronize()
        loader.synchronize()

    run(2)
    n = max(1, args.steps)
    t0 = time.perf_counter()
    run(n)
    dt = (time.perf_counter() - t0) / n
    h2d = Wh.numel() * 2 + Xh.numel() * 2
    d2h = sum(o.numel() for o in outs.values()) + sum(t.numel() * 4 for t in touts.values())
    return {"value": round(5 * R * C / dt / 1e6, 2), "unit": "M elem/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 3),
            "pipelining": "inputs of step k+1 copied during step k (double-buffered); outputs copied "
                          "back during the next format's encode"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--only", default=None,
                    help="run one part of the step alone and print its time (for profiling runs)")
    args = ap.parse_args()
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
