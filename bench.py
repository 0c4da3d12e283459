"""Benchmark of one DSpark round (draft -> schedule -> verify) on GB300.

Default workload: the DeepSeek-scale configuration (R = 128 requests,
gamma = 16, V = 129280, Markov rank 256, bf16, temperature 1, causal
scheduler), synthetic inputs from the seeded generators, built on the device.

One "step" is one whole round through the library's public C ABI
(dspark_round). `value` is drafted positions per second (R * gamma / round
latency) from CUDA events on the launching stream, inputs resident in HBM,
L2 flushed (256 MiB write) between steps outside the timed events. `e2e`
is the same metric through the same C ABI with the step's inputs copied from
pinned host memory and the results copied back inside the timed region.

--impl reference times the oracle (the plain CPU implementation) on a bounded
sample of the same workload on the host cores.

One step at N = 1 replays the round captured as a CUDA graph (direct calls
are timed beside it).

Multi-GPU: the path shards by request. Under torchrun every rank drafts and
verifies its own requests on its own GPU; the confidences are all-gathered
(NCCL) and every rank runs the same global schedule over the whole batch
(speculative_decoding_draft_seq_gb300/shard.py). Timing is the max over ranks
and `value` sums all ranks' positions.
"""
import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft+verify round latency (µs) & positions/s at R=128,γ=16,V=129280; %HBM roof"
FALLBACK_HBM = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM, "fallback"


def bf16_peak_tflops():
    """Dense bf16 peak for a kernel timed alone (the burst figure)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured bf16_tflops (burst)"
    return 1900.0, "fallback"


def algorithmic_bytes(cfg, L):
    """Bytes each pass must touch once (re-reads excluded)."""
    e = 2 if cfg.dtype == "bf16" else 4
    draft = cfg.R * cfg.gamma * cfg.V * e + cfg.rank * cfg.V * e + cfg.R * cfg.gamma * cfg.rank * e
    verify = int((L + 1).sum()) * cfg.V * e
    return draft, verify


def cpu_baseline(cfg, n_req, steps=1, warmup=0, timeout=900):
    """Times the oracle in one single-threaded child process: `warmup` untimed
    and `steps` timed steps, each a full round over all requests' schedule with
    draft + verify of `n_req` requests (a different sample every step)."""
    code = (
        "import time, json, sys; sys.path.insert(0, %r)\n"
        "import workloads as W\n"
        "from oracle.round import run_round\n"
        "cfg = W.CONFIGS[%r]\n"
        "n, steps, warm = %d, %d, %d\n"
        "pool = min(cfg.R, max(n, 8))\n"
        "reqs = [[(i * n + j) %% pool for j in range(n)] for i in range(steps + warm)]\n"
        "allr = sorted(set(r for q in reqs for r in q))\n"
        "inp = W.oracle_inputs(cfg, allr)\n"
        "ts = []\n"
        "for i, q in enumerate(reqs):\n"
        "    t = time.perf_counter(); run_round(inp, requests=q); dt = time.perf_counter() - t\n"
        "    if i >= warm: ts.append(dt)\n"
        "print(json.dumps({'seconds': ts}))\n" % (ROOT, cfg.name, n_req, steps, warmup))
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=timeout)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    ts = json.loads(out.stdout.strip().splitlines()[-1])["seconds"]
    dt = float(sum(ts))
    pos = n_req * cfg.gamma * len(ts)
    return {"value": pos / dt, "unit": "positions/s", "cores": 1, "kind": "oracle",
            "host": {"nproc": os.cpu_count(), "cpu": host_cpu_model()},
            "sample": f"{len(ts)} step(s) of {n_req} of {cfg.R} requests x gamma={cfg.gamma} (drawn from the "
                      f"first {min(cfg.R, max(n_req, 8))}; each a full round: "
                      f"schedule over all requests, draft + verify of the sampled ones), single thread, "
                      f"{dt:.1f} s timed"}


def host_cpu_model():
    """The host CPU's model name (from /proc/cpuinfo; Arm hosts report implementer and part)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in info:
            if line.split(":")[0].strip() == key:
                return line.split(":", 1)[1].strip()
    return "unknown"


class ClockSampler:
    """SM clock, power and clock-event reasons sampled during the timed region.

    Reads NVML directly (ctypes on the driver's libnvidia-ml) from a background
    thread about once a millisecond, so that even a timed region of a few
    milliseconds gets several samples; falls back to `nvidia-smi -lms 25` when
    NVML cannot be loaded. Only reads: no clock or other setting is touched.
    Each sample is written to clocks_rank<r>.csv in $DSPARK_OUT_DIR (or runs/)."""
    # clock-event reason bits of NVML
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self):
        self.proc = None
        self.path = None
        self.thread = None
        self.rows = []
        self.max_mhz = None

    def _nvml_handle(self, index):
        import ctypes
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                pass
        if lib is None or lib.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        try:  # the device this process runs on, by PCI address (NVML's index order may differ from CUDA's)
            import torch
            pr = torch.cuda.get_device_properties(torch.cuda.current_device())
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0:
                return lib, h
        except Exception:
            pass
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)) != 0:
            return None, None
        return lib, h

    def start(self, rank):
        import threading
        out_dir = os.environ.get("DSPARK_OUT_DIR", os.path.join(ROOT, "runs"))
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, f"clocks_rank{rank}.csv")
        dev = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0] or "0"
        index = int(dev) if dev.isdigit() else rank
        lib, h = self._nvml_handle(index)
        if lib is None:
            return self._start_smi(index)
        import ctypes
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.stop_flag = threading.Event()

        def loop():
            clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            while not self.stop_flag.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    p_ok = lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0
                    r_ok = get_reasons(h, ctypes.byref(rs)) == 0
                    self.rows.append((time.time(), float(clk.value), pw.value / 1000.0 if p_ok else None,
                                      int(rs.value) if r_ok else 0))
                time.sleep(0.001)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()
        t0 = time.time()  # the first sample exists before the timed region starts
        while not self.rows and time.time() - t0 < 2.0:
            time.sleep(0.001)

    def _start_smi(self, index):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "25"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()  # nvidia-smi needs a moment before its first line
        while time.time() - t0 < 5.0:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join()
            rows = self.rows
            if not rows:
                return None
            with open(self.path, "w") as f:
                f.write("time_s,sm_mhz,power_w,reasons_mask\n")
                for t, c, pw, rs in rows:
                    f.write(f"{t:.6f},{c:.0f},{'' if pw is None else f'{pw:.1f}'},{rs:#x}\n")
            sm = sorted(r[1] for r in rows)
            reasons = sorted({n for r in rows for bit, n in self.REASONS.items() if r[3] & bit})
            return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": self.max_mhz, "reasons": reasons,
                    "samples": len(rows), "source": "nvml"}
        if self.proc is None:
            return None
        self.proc.terminate()
        self.proc.wait()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        if not rows:
            return None
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows), "source": "nvidia-smi"}


# DRAM bytes per launch of the persistent drafting / residual kernel, from
# one ncu capture of the full-size round (profiles/traffic_ds_round.md). The
# figure stands only while the CUDA sources are the ones it was taken on.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_ds_round.md")


def label_bytes(cfg):
    """Distinct bytes the acceptance-label pass must read: target rows 0..gamma-1, the base
    rows, W2 once and the W1 rows of the drafted tokens."""
    e = 2 if cfg.dtype == "bf16" else 4
    return (2 * cfg.R * cfg.gamma * cfg.V + cfg.rank * cfg.V + cfg.R * cfg.gamma * cfg.rank) * e


# The sources the kernels with recorded DRAM traffic (the drafting sweep and its residual mode) are
# compiled from: a change to any of them voids the record; host-only files (api.cu, the header's
# declarations) do not.
TRAFFIC_SOURCES = ("common.cuh", "draft_persistent.cu", "internal.h", "sched_common.cuh", "tc_ptx.cuh",
                   "verify_common.cuh")


def csrc_digest():
    import hashlib
    d = os.path.join(ROOT, "speculative_decoding_draft_seq_gb300", "csrc")
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()


def measured_traffic(kernel):
    key = {"draft": "traffic.draft", "verify": "traffic.verify_resid"}[kernel]
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    vals = dict(l.split()[:2] for l in lines if len(l.split()) >= 2 and l.split()[0].startswith(("traffic.", "sources")))
    if vals.get("sources") != csrc_digest() or key not in vals:
        return None
    return int(vals[key])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="ds")
    ap.add_argument("--temperature", type=float, default=None)
    ap.add_argument("--cpu-requests", type=int, default=48)
    ap.add_argument("--no-graph", action="store_true", help="time direct dspark_round calls, no CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gamma", type=int, default=None, help="override the workload's draft length")
    ap.add_argument("--profile", choices=["round", "draft", "gated", "lm_head"], default=None,
                    help="launch only, for an ncu capture: 'round' = one round then two verify calls, "
                         "'draft' = three drafting calls, 'gated' = three gated-head drafting calls, "
                         "'lm_head' = three base-logit GEMMs at d = 7168 over 16,384 vocabulary columns; "
                         "prints the device status")
    args = ap.parse_args()

    import workloads as W
    cfg = W.CONFIGS[args.config]
    if args.temperature is not None:
        cfg = W.with_(cfg, T=args.temperature)
    if args.gamma is not None:
        cfg = W.with_(cfg, gamma=args.gamma)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    workload = (f"{cfg.name}: R={cfg.R} gamma={cfg.gamma} V={cfg.V} rank={cfg.rank} {cfg.dtype} "
                f"T={cfg.T} scheduler={['causal', 'lagged', 'all'][cfg.mode]}")

    if args.impl == "reference":
        if rank != 0:
            return
        # one request per step: the oracle takes about a quarter of a second per
        # DeepSeek-scale request, so the default 300 steps stay within minutes
        b = cpu_baseline(cfg, 1, steps=max(1, args.steps), warmup=args.warmup)
        v = b["value"]
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "positions/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * cfg.R * cfg.gamma / v, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": workload},
                "cpu_baseline": {"value": v, "unit": "positions/s", "cores": 1, "kind": "oracle",
                                 "sample": b["sample"], "host": b["host"]},
                "e2e": {"value": v, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import numpy as np
    import torch
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_draft_seq_gb300 import dspark

    # each rank holds its own R requests (its own seed); with several ranks the scheduler ranks all
    # ranks' requests against one table of world x the single-GPU size (see shard.py)
    inp = W.device_inputs(W.with_(cfg, seed=cfg.seed + 101 * rank) if world > 1 else cfg, dev)
    R, gamma, V = cfg.R, cfg.gamma, cfg.V
    dt_code = dspark.BF16 if cfg.dtype == "bf16" else dspark.FP32
    ws = dspark.new_workspace(R, gamma, V, cfg.rank, dt_code, cfg.n_table, dev)
    out = dspark.RoundOutputs(R, gamma, dev)
    stream = torch.cuda.current_stream()
    sharded = None
    if world > 1:
        from speculative_decoding_draft_seq_gb300.shard import ShardedRound
        cfg_all = W.with_(cfg, R=cfg.R * world, n_table=cfg.n_table * world)
        inp["sps"] = torch.from_numpy(W.sps_table(cfg_all)).to(dev)
        sharded = ShardedRound(dspark, R, gamma, V, cfg.rank, dt_code, cfg_all.n_table, dev)
    if args.profile:
        if args.profile == "round":
            dspark.round_(inp["base"], inp["target"], inp["anchor"], inp["W1"], inp["W2"], inp["conf"],
                          inp["conf_lag"], inp["sps"], inp["mode"], inp["T"], inp["seed"], out, ws)
            for _ in range(2):
                dspark.verify(inp["target"], inp["base"], inp["anchor"], inp["W1"], inp["W2"], out.tokens,
                              out.q_tok, out.q_stats, out.sched_len, inp["T"], inp["seed"], out.out_tokens,
                              out.accepted_len, out.p_tok, ws)
        elif args.profile == "draft":
            for _ in range(3):
                dspark.draft_sequential(inp["base"], inp["anchor"], inp["W1"], inp["W2"], inp["T"], inp["seed"],
                                        out.tokens, out.q_tok, out.q_stats, ws)
        elif args.profile == "gated":
            gate = W.gate_device(W.with_(cfg, gated=True), dev)
            for _ in range(3):
                dspark.draft_sequential_gated(inp["base"], inp["anchor"], inp["W1"], gate, inp["W2"], inp["T"],
                                              inp["seed"], out.tokens, out.q_tok, out.q_stats, ws)
        else:  # a slice of the vocabulary keeps the capture small (LM head 235 MB, larger than L2)
            cfg_h = W.with_(cfg, V=16384)
            H = W.hidden_device(cfg_h, 7168, dev)
            LMW = W.lm_head_device(cfg_h, 7168, dev)
            o = torch.empty((R, gamma, 16384), dtype=torch.bfloat16, device=dev)
            for _ in range(3):
                dspark.lm_head(H, LMW, o, ws)
        torch.cuda.synchronize()
        st = dspark.device_status(ws)
        print(json.dumps({"profile": args.profile, "workload": workload, "status": dspark.status_string(st)}))
        if st != dspark.OK:
            sys.exit(1)
        return
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def one_round():
        if sharded is not None:  # draft, all-gather of confidences + global schedule, verify
            sharded(inp, out)
            return
        dspark.round_(inp["base"], inp["target"], inp["anchor"], inp["W1"], inp["W2"], inp["conf"],
                      inp["conf_lag"], inp["sps"], inp["mode"], inp["T"], inp["seed"], out, ws)

    for _ in range(max(3, args.warmup)):
        one_round()
    torch.cuda.synchronize()
    st = dspark.device_status(ws)
    if st != dspark.OK:
        raise RuntimeError(f"device status {dspark.status_string(st)}")
    launches_per_round = dspark.last_launch_count()

    # stage timing (draft / schedule / verify separately, same stream)
    def time_stage(fn, n):
        ts = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return float(np.median(ts))

    t_draft = time_stage(lambda: dspark.draft_sequential(inp["base"], inp["anchor"], inp["W1"], inp["W2"],
                                                         inp["T"], inp["seed"], out.tokens, out.q_tok,
                                                         out.q_stats, ws), max(3, args.steps // 4))
    t_sched = time_stage(lambda: dspark.schedule(inp["conf"], inp["conf_lag"], inp["sps"], inp["mode"],
                                                 out.sched_len, out.K, out.tau_theta, ws),
                         max(3, args.steps // 4))
    t_verify = time_stage(lambda: dspark.verify(inp["target"], inp["base"], inp["anchor"], inp["W1"],
                                                inp["W2"], out.tokens, out.q_tok, out.q_stats, out.sched_len,
                                                inp["T"], inp["seed"], out.out_tokens, out.accepted_len,
                                                out.p_tok, ws), max(3, args.steps // 4))
    # the acceptance-label pass (training signal of the confidence head; not part of the round)
    labels = torch.empty((R, gamma), dtype=torch.float32, device=dev)
    try:  # the sampled form needs the tensor-core shape
        t_labels = time_stage(lambda: dspark.acceptance_labels(inp["target"], inp["base"], inp["anchor"], inp["W1"],
                                                               inp["W2"], out.tokens, out.q_stats, inp["T"], labels,
                                                               ws), max(3, args.steps // 8))
    except dspark.DSparkError:
        t_labels = None

    # Sequential Temperature Scaling (offline calibration of the confidences): a held-out set of
    # 65,536 blocks x gamma drawn from over-confident scores, 64 grid temperatures, 15 bins
    n_sts = 65536
    g_sts = torch.Generator(device="cpu").manual_seed(7)
    z_sts = torch.randn((n_sts, gamma), generator=g_sts, dtype=torch.float64) * 1.5 + 1.0
    c_sts = torch.sigmoid(z_sts).float().to(dev)
    passed = torch.rand((n_sts, gamma), generator=g_sts, dtype=torch.float64) < torch.sigmoid(0.6 * z_sts)
    first_fail = torch.where(passed.all(dim=1), torch.full((n_sts,), gamma), (~passed).int().argmax(dim=1))
    a_sts = first_fail.int().to(dev)
    grid_sts = torch.exp(torch.linspace(np.log(0.25), np.log(4.0), 64, dtype=torch.float64)).float().to(dev)
    t_sts = torch.zeros(gamma, dtype=torch.float32, device=dev)
    t_sts_fit = time_stage(lambda: dspark.sts_fit(c_sts, a_sts, grid_sts, 15, t_sts), 3)
    conf_cal = torch.empty_like(inp["conf"])
    t_sts_apply = time_stage(lambda: dspark.sts_apply(inp["conf"], t_sts, conf_cal), 5)

    # the hidden-state path: base logits from the backbone's hidden states and the LM head
    # (tensor cores), then the sequential draft on them; d = 7168 (DeepSeek hidden size)
    hidden_path = None
    if cfg.dtype == "bf16":
        d_h = 7168
        H = W.hidden_device(cfg, d_h, dev)
        LMW = W.lm_head_device(cfg, d_h, dev)
        base_h = torch.empty_like(inp["base"])
        t_lm = time_stage(lambda: dspark.lm_head(H, LMW, base_h, ws), 5)
        t_lm_draft = time_stage(lambda: (dspark.lm_head(H, LMW, base_h, ws),
                                         dspark.draft_sequential(base_h, inp["anchor"], inp["W1"], inp["W2"], inp["T"],
                                                                 inp["seed"], out.tokens, out.q_tok, out.q_stats, ws)), 3)
        if dspark.device_status(ws) != dspark.OK:
            raise RuntimeError("device status after the hidden-state path")
        flops = 2.0 * R * gamma * d_h * V
        bf16_peak, bf16_kind = bf16_peak_tflops()
        hidden_path = {"d": d_h, "lm_head_us": t_lm * 1e3, "tflops": flops / (t_lm * 1e-3) / 1e12,
                       "peak_tflops": bf16_peak, "peak_kind": bf16_kind,
                       "frac": flops / (t_lm * 1e-3) / 1e12 / bf16_peak,
                       "lm_head_plus_draft_us": t_lm_draft * 1e3,
                       "h2d_bytes_hidden": H.numel() * 2, "h2d_bytes_base_logits": inp["base"].numel() * 2}
        del base_h  # H and the LM head stay for the hidden-state end-to-end run below

    # the recurrent (gated) head: the same workload with a gate table [V, rank]
    gated = None
    if cfg.dtype == "bf16":
        gate = W.gate_device(W.with_(cfg, gated=True), dev)
        gout = dspark.RoundOutputs(R, gamma, dev)
        try:
            t_gdraft = time_stage(lambda: dspark.draft_sequential_gated(
                inp["base"], inp["anchor"], inp["W1"], gate, inp["W2"], inp["T"], inp["seed"], gout.tokens,
                gout.q_tok, gout.q_stats, ws), max(3, args.steps // 8))
            t_ground = time_stage(lambda: dspark.round_gated(
                inp["base"], inp["target"], inp["anchor"], inp["W1"], gate, inp["W2"], inp["conf"],
                inp["conf_lag"], inp["sps"], inp["mode"], inp["T"], inp["seed"], gout, ws), max(3, args.steps // 8))
            if dspark.device_status(ws) != dspark.OK:
                raise RuntimeError("device status after the gated rounds")
            gb = algorithmic_bytes(cfg, np.zeros(R, dtype=np.int64))[0] + R * gamma * cfg.rank * 2  # + gate rows
            gated = {"round_us": t_ground * 1e3, "draft_us": t_gdraft * 1e3, "draft_algorithmic_bytes": gb,
                     "draft_frac": gb / (t_gdraft * 1e-3) / 1e9 / peaks()[0]}
        except dspark.DSparkError:
            gated = None

    # the full-verification bound: the same round with the scheduler in ALL mode, every drafted
    # position verified (R * (gamma + 1) target rows), as the pages' offline evaluation runs it
    full_verify = None
    if world == 1:
        fout = dspark.RoundOutputs(R, gamma, dev)
        n_fv = max(3, args.steps // 8)
        t_fround = time_stage(lambda: dspark.round_(
            inp["base"], inp["target"], inp["anchor"], inp["W1"], inp["W2"], inp["conf"], inp["conf_lag"],
            inp["sps"], W.ALL, inp["T"], inp["seed"], fout, ws), n_fv)
        t_fverify = time_stage(lambda: dspark.verify(
            inp["target"], inp["base"], inp["anchor"], inp["W1"], inp["W2"], fout.tokens, fout.q_tok,
            fout.q_stats, fout.sched_len, inp["T"], inp["seed"], fout.out_tokens, fout.accepted_len, fout.p_tok,
            ws), n_fv)
        if dspark.device_status(ws) != dspark.OK:
            raise RuntimeError("device status after the full-verification rounds")
        Lf = fout.sched_len.cpu().numpy()
        Af = fout.accepted_len.cpu().numpy()
        bvf = algorithmic_bytes(cfg, Lf)[1]
        full_verify = {"mode": "all", "round_us": t_fround * 1e3, "verify_us": t_fverify * 1e3,
                       "verify_algorithmic_bytes": bvf,
                       "verify_frac": bvf / (t_fverify * 1e-3) / 1e9 / peaks()[0],
                       "scheduled_positions": int(Lf.sum()), "emitted": int((Af + 1).sum())}
        del fout

    # the round as a CUDA graph (its launches and memsets replayed as one unit, as a serving
    # loop would run it); the direct call is timed beside it
    graph, graph_note = None, None
    if not args.no_graph and world == 1:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                one_round()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                one_round()
            graph.replay()
            torch.cuda.synchronize()
            if dspark.device_status(ws) != dspark.OK:
                raise RuntimeError("device status after the graph replay")
        except Exception as e:  # capture not possible here: time the direct call only
            graph, graph_note = None, f"graph capture failed: {type(e).__name__}"
            torch.cuda.synchronize()

    def timed(fn, n):
        ts = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return ts

    direct_ms = float(np.mean(timed(one_round, max(3, args.steps // 4)))) if graph is not None else None
    clocks = ClockSampler()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start(rank)
    times = timed(graph.replay if graph is not None else one_round, args.steps)
    pct = {q: float(np.percentile(times, q)) * 1e3 for q in (10, 50, 90)}
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = float(np.sum(times)) / args.steps
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    value = world * R * gamma / (ms * 1e-3)
    # the timed rounds' lengths (the end-to-end legs below write into `out` too)
    L = out.sched_len.cpu().numpy()
    A = out.accepted_len.cpu().numpy()

    # end to end through the same C ABI from pinned host buffers
    host = {k: inp[k].cpu().pin_memory() for k in ("base", "target", "anchor", "conf") }
    if inp["conf_lag"] is not None:
        host["conf_lag"] = inp["conf_lag"].cpu().pin_memory()
    # two slots of device inputs and outputs: while the round of step i runs on `stream`, the
    # inputs of step i + 1 are copied on a copy stream (as a serving loop would overlap them);
    # every step's copies in and out are inside the timed region. Of the target logits only the
    # rows verification reads are sent (rows 0..L_r, dspark_copy_scheduled_rows): the step's
    # confidences go first, the scheduler runs on them on its own workspace while the previous
    # round computes, and its lengths come back to the host to pick the rows. With `lm`, the
    # step sends the backbone's hidden states instead of base logits and the base logits are
    # computed on the device with the LM head (dspark_lm_head) before the round.
    res_keys = ("out_tokens", "accepted_len", "sched_len")
    outs = [out, dspark.RoundOutputs(R, gamma, dev)]
    res_host = [{k: torch.empty_like(getattr(o, k), device="cpu").pin_memory() for k in res_keys} for o in outs]
    ws_ahead = dspark.new_workspace(R, gamma, 1, cfg.rank, dt_code, cfg.n_table, dev)
    L_dev = torch.empty(R, dtype=torch.int32, device=dev)
    K_dev = torch.empty(1, dtype=torch.int32, device=dev)
    tt_dev = torch.empty(2, dtype=torch.float64, device=dev)
    L_host = torch.empty(R, dtype=torch.int32).pin_memory()
    copy_stream, sched_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined_e2e(host_in, n, lm=None):
        small = [k for k in host_in if k != "target"]
        conf_keys = [k for k in ("conf", "conf_lag") if k in host_in]
        dev_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host_in.items()} for _ in range(2)]
        base_dev = [torch.empty_like(inp["base"]) for _ in range(2)] if lm is not None else None
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        conf_in, L_back = torch.cuda.Event(), torch.cuda.Event()
        sent = {"target": 0}

        def copy_in(j):
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[j])  # the round that last used slot j has read it
                # the confidences first: the look-ahead schedule and the host's choice of target rows
                # then overlap the base-logit copy, and the row copies queue right behind it
                for k in conf_keys:
                    dev_in[j][k].copy_(host_in[k], non_blocking=True)
                conf_in.record(copy_stream)
                for k in small:
                    if k not in conf_keys:
                        dev_in[j][k].copy_(host_in[k], non_blocking=True)
            if sharded is None:
                sched_stream.wait_event(conf_in)
                dspark.schedule(dev_in[j]["conf"], dev_in[j].get("conf_lag"), inp["sps"], inp["mode"], L_dev,
                                K_dev, tt_dev, ws_ahead, stream=sched_stream)
                with torch.cuda.stream(sched_stream):
                    L_host.copy_(L_dev, non_blocking=True)
                    L_back.record(sched_stream)
                L_back.synchronize()  # the host picks the rows (the GPU keeps running the current round)
            else:  # the global schedule needs every rank's confidences: send every target row
                L_host.fill_(gamma)
            dspark.copy_scheduled_rows(host_in["target"], dev_in[j]["target"], L_host, stream=copy_stream)
            sent["target"] = int((L_host.clamp(0, gamma) + 1).sum()) * V * host_in["target"].element_size()
            copied[j].record(copy_stream)

        def compute(j):
            stream.wait_event(copied[j])
            d = dev_in[j]
            base = d["base"] if lm is None else base_dev[j]
            if lm is not None:
                dspark.lm_head(d["hidden"], lm, base, ws)
            if sharded is not None:  # local draft and verify, all-gathered confidences, global schedule
                sharded(dict(inp, base=base, target=d["target"], anchor=d["anchor"], conf=d["conf"],
                             conf_lag=d.get("conf_lag")), outs[j])
            else:
                dspark.round_(base, d["target"], d["anchor"], inp["W1"], inp["W2"], d["conf"], d.get("conf_lag"),
                              inp["sps"], inp["mode"], inp["T"], inp["seed"], outs[j], ws)
            consumed[j].record(stream)
            for k, v in res_host[j].items():
                v.copy_(getattr(outs[j], k), non_blocking=True)

        def run(m):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(copy_stream)
            copy_in(0)
            for i in range(m):
                compute(i % 2)
                if i + 1 < m:
                    copy_in((i + 1) % 2)
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b) / m

        run(2)
        torch.cuda.synchronize()
        ms_step = run(n)
        h2d_b = sum(host_in[k].numel() * host_in[k].element_size() for k in small) + sent["target"]
        d2h_b = sum(v.numel() * v.element_size() for v in res_host[0].values()) + L_host.numel() * 4
        return ms_step, h2d_b, d2h_b

    e2e_ms, h2d, d2h = pipelined_e2e(host, max(3, args.steps // 2))
    if hidden_path is not None:  # the same loop sending hidden states (the LM head on the device)
        host_h = {k: v for k, v in host.items() if k != "base"}
        host_h["hidden"] = H.cpu().pin_memory()
        h_ms, h_h2d, h_d2h = pipelined_e2e(host_h, max(3, args.steps // 8), lm=LMW)
        if dspark.device_status(ws) != dspark.OK:
            raise RuntimeError("device status after the hidden-state end-to-end run")
        hidden_path["e2e"] = {"value": world * R * gamma / (h_ms * 1e-3), "unit": "positions/s",
                              "h2d_bytes_per_step": h_h2d, "d2h_bytes_per_step": h_d2h, "ms_per_step": h_ms}
        del H, LMW, host_h

    peak, peak_kind = peaks()
    bd, bv = algorithmic_bytes(cfg, L)
    draft_gbs = bd / (t_draft * 1e-3) / 1e9
    verify_gbs = bv / (t_verify * 1e-3) / 1e9
    dominant = "draft" if t_draft >= t_verify else "verify"
    ach = draft_gbs if dominant == "draft" else verify_gbs
    traffic = measured_traffic(dominant)
    line = {
        "metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "round_us": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": workload, "l2": "flushed between steps (256 MiB write, outside the events)",
                   "parallelism": (f"request-sharded x{world}: local draft and verify, all-gathered "
                                   f"confidences, global schedule") if world > 1 else "single GPU",
                   "launch": "CUDA graph of one dspark_round call, replayed per step" if graph is not None
                   else (graph_note or "direct dspark_round call per step")},
        "round_us_direct_call": None if direct_ms is None else direct_ms * 1e3,
        "round_us_p10_median_p90": [pct[10], pct[50], pct[90]],
        "stages_us": {"draft": t_draft * 1e3, "schedule": t_sched * 1e3, "verify": t_verify * 1e3},
        "stages_note": ("each entry point timed alone (verify: its row-statistics launch and its residual "
                        "launch; roofline.verify_frac is this standalone call); inside dspark_round one extra "
                        "CTA of the drafting launch computes the schedule and a few more stream the scheduled "
                        "target rows' statistics while the other CTAs sweep, its sweep CTAs run the acceptance "
                        "chains after the last draw, and the residual draw is the round's second launch"),
        "sts": {"fit_us": t_sts_fit * 1e3, "fit_rows": n_sts, "grid": 64, "bins": 15,
                "apply_us": t_sts_apply * 1e3},
        "gated_head": gated,
        "full_verify": full_verify,
        "hidden_path": hidden_path,
        "labels": None if t_labels is None else {
            "us": t_labels * 1e3, "algorithmic_bytes": label_bytes(cfg),
            "achieved_gbs": label_bytes(cfg) / (t_labels * 1e-3) / 1e9,
            "frac": label_bytes(cfg) / (t_labels * 1e-3) / 1e9 / peak},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": ach, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s", "frac": ach / peak,
                     "traffic": traffic,
                     "algorithmic_bytes": bd if dominant == "draft" else bv,
                     "draft_frac": draft_gbs / peak, "verify_frac": verify_gbs / peak},
        "round_stats": {"scheduled_positions": int(L.sum()), "accepted": int(A.sum()),
                        "emitted": int((A + 1).sum()),
                        "scheduled_positions_per_s": world * int(L.sum()) / (ms * 1e-3),
                        "emitted_tokens_per_s": world * int((A + 1).sum()) / (ms * 1e-3)},
        "e2e": {"value": world * R * gamma / (e2e_ms * 1e-3), "unit": "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "overlap": "step i+1's host-to-device copies run during step i's round (two input slots)",
                "target_rows": "only rows 0..L_r of each request (those verification reads), picked by a "
                               "look-ahead schedule of the step's confidences"},
        "clocks": clk,
        "gpu_launches": launches_per_round * args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_requests)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
