"""Benchmark: decode tokens/s and µs/token of the single-launch decode
MegaKernel on one GB300, with its HBM-roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the CPU oracle on the host cores

A step is one decode step of the whole stack plus LM head (one kernel
launch) for the workload's batch.  Steps walk the workload's decode window
(positions ctx .. ctx + steps_of_workload - 1) and wrap around it, so every
timed step has the workload's context length.  Inputs (weights, KV cache,
tokens) are seeded, synthetic and resident in HBM before timing; the weights
alone are larger than L2, so no flush is needed between steps.

Under torchrun (N > 1) every rank runs an independent replica (the decode
step does not shard: replicas only); the value is the tokens of all ranks
divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s & µs/token at batch 1 (1 GB300); % of 8 TB/s HBM roofline"
DEFAULT_WORKLOAD = "tinyllama_1b1"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["persistent_sm_decode_gb300/csrc/amk_kernel.cu", "persistent_sm_decode_gb300/csrc/amk_internal.h"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(mp["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_bytes(wl, position: int, batch: int) -> int:
    """Algorithmic HBM bytes of one decode step: every linear weight (+ int8
    scales) and norm gain once, one embedding row per sequence, K and V of
    positions 0..p-1 read, K and V of slot p written, fp32 logits written."""
    kv = batch * wl.n_layers * wl.n_kv_heads * wl.head_dim * 2 * 2 * (position + 1)
    return wl.weight_bytes() + batch * wl.hidden * 2 + kv + batch * wl.vocab * 4


class NvmlClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, read through
    NVML every millisecond or so on a host thread while the timed region
    runs: a decode step takes well under a millisecond, so nvidia-smi's
    sampling interval would see a whole timed region at most once.  Only
    reads; no GPU setting is changed."""
    # nvmlClocksEventReasons bits (nvml.h): sw power cap, hw slowdown, sw thermal, hw thermal
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            import ctypes
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            # CUDA's ordinal and NVML's index differ under CUDA_VISIBLE_DEVICES: find the GPU by the
            # PCI address of the CUDA device
            import torch
            pr = torch.cuda.get_device_properties(gpu_index)
            bus = None
            if all(hasattr(pr, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
                bus = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            if bus is None or self.nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[gpu_index]) if vis and all(
                    x.strip().isdigit() for x in vis.split(",")) else gpu_index
                if self.nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h)) != 0:
                    return
            self.c_uint, self.c_ull, self.byref = ctypes.c_uint, ctypes.c_ulonglong, ctypes.byref
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 \
                else None
            self.ok = True
        except Exception:
            self.ok = False

    def _read(self):
        while not self._stop.is_set():
            clk, rs = self.c_uint(), self.c_ull()
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, self.byref(clk)) == 0 and \
                    self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, self.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self.t.join(timeout=2)

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _c, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _r in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """nvidia-smi samples of the GPU clocks and throttle reasons while running
    (the fallback where NVML cannot be loaded)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(x: float, dist, device: str) -> float:
    """The largest x over all ranks (x itself without a process group): every
    replica's timed region ends together only when the slowest one does."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, batch: int, steps: int, seconds: float) -> float:
    """Tokens of every replica per second of the slowest one."""
    return world * batch * steps / seconds


def cpu_model() -> str:
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def time_oracle(model, kc, vc, wl, budget_s: float, max_steps: int, threads: int = 0):
    """The oracle as it stands on the host cores (``threads`` of them, 0: all):
    decode steps of the workload until the budget or max_steps is reached.
    Returns (tokens/s, steps, threads, seconds)."""
    import numpy as np
    import oracle
    if threads:
        every = oracle.num_threads()
        oracle.set_num_threads(threads)
        try:
            return time_oracle(model, kc, vc, wl, budget_s, max_steps)
        finally:
            oracle.set_num_threads(every)
    orc = oracle.Oracle(model, kc, vc)
    B = kc.shape[1]
    tok = np.array([(1 + 7919 * b) % wl.vocab for b in range(B)], dtype=np.int32)
    t0 = time.perf_counter()
    n = 0
    while n < max_steps:
        lg = orc.step(tok, np.full(B, wl.ctx + (n % wl.steps), dtype=np.int32))
        tok = np.argmax(lg, axis=1).astype(np.int32)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return B * n / dt, n, oracle.num_threads(), dt


def traffic_from_profile(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        e = t.get(workload)
        if e and e.get("kernel_sha") == kernel_hash():
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def reference_arm(args, wl, rank, world):
    """The oracle on host cores, on this arm's config/metric/unit."""
    if rank != 0:
        return 0
    import numpy as np
    import synth
    model = synth.make_model(wl, seed=1)
    kc, vc = synth.make_kv(wl, seed=2)
    # warm-up steps, then the timed ones, within a few minutes in total
    time_oracle(model, kc, vc, wl, budget_s=10.0, max_steps=args.warmup)
    tps, n, threads, dt = time_oracle(model, kc, vc, wl, budget_s=90.0, max_steps=args.steps)
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * dt / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(wl),
            "cpu_baseline": {"kind": "oracle", "value": tps, "unit": "tokens/s", "cores": threads,
                             "sample": "%d of %d requested decode steps of %s timed (%.1f s budget) on %s"
                                       % (n, args.steps, wl.name, 90.0, cpu_model())},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_block(wl):
    return {"workload": wl.name, "batch": wl.batch, "context": wl.ctx, "decode_window": wl.steps,
            "shape": "L%d H%d q%d kv%d d%d I%d V%d %s%s" % (wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads,
                                                        wl.head_dim, wl.intermediate, wl.vocab, wl.weight_dtype,
                                                        " tied" if wl.tied else ""),
            "l2": "weights %.2f GB per step > 129 MB L2: no flush needed" % (wl.weight_bytes() / 1e9)}


def workload_dtype(wl) -> str:
    """The arithmetic the path computes in: bf16 products with fp32 sums, or
    int8 / int4 weights times bf16 activations (W8A16 / W4A16) with fp32 sums."""
    return {"int8": "int8xbf16", "int4": "int4xbf16"}.get(wl.weight_dtype, "bf16")


def device_model(wl, seed: int):
    """Weights of a workload's shape filled on the device by torch's seeded
    generator, with the synthetic recipe's distributions (bf16 N(0, 0.02);
    int8 uniform on [-127, 127] with row scales 0.02/127; norm gains 1.0).
    Only the timing sub-records use these: the decode step's time does not
    depend on the values, and drawing a 7B-shaped model on the host takes a
    minute.  Parity tests always use the host generator's bits."""
    import torch
    from synth import mat_shapes
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    H, V = wl.hidden, wl.vocab

    def mat(shape):
        if wl.weight_dtype == "int4":
            codes = torch.randint(0, 256, (shape[0], shape[1] // 2), generator=g, device="cuda",
                                  dtype=torch.int32).to(torch.uint8)
            return codes, torch.full((shape[0], shape[1] // wl.group_size), wl.weight_std / 7.0, device="cuda",
                                     dtype=torch.float32)
        if wl.weight_dtype == "int8":
            q = torch.randint(-127, 128, shape, generator=g, device="cuda", dtype=torch.int8)
            return q, torch.full((shape[0],), wl.weight_std / 127.0, device="cuda", dtype=torch.float32)
        return (torch.randn(shape, generator=g, device="cuda") * wl.weight_std).to(torch.bfloat16), None

    ones = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    keys = {"wq": "s_q", "wk": "s_k", "wv": "s_v", "wo": "s_o", "w_gate": "s_gate", "w_up": "s_up",
            "w_down": "s_down"}
    layers = []
    for _ in range(wl.n_layers):
        d = {"attn_norm": ones.clone(), "mlp_norm": ones.clone()}
        for m, shape in mat_shapes(wl).items():
            q, sc = mat(shape)
            d[m] = q
            if sc is not None:
                d[keys[m]] = sc
        layers.append(d)
    embed = (torch.randn((V, H), generator=g, device="cuda") * wl.weight_std).to(torch.bfloat16)
    lm, s_lm = (None, None) if wl.tied else mat((V, H))
    return {"embed": embed, "final_norm": ones.clone(), "layers": layers, "lm_head": lm, "s_lm": s_lm}


def device_kv(wl, seed: int, batch: int):
    """K then V cache [2][L][B][nkv][Smax][d] bf16 on the device: N(0, 1) at
    the positions below the workload's context, zero above (timing only)."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    kv = torch.zeros((2, wl.n_layers, batch, wl.n_kv_heads, wl.max_seq, wl.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    for l in range(wl.n_layers):
        kv[:, l, :, :, : wl.ctx] = torch.randn((2, batch, wl.n_kv_heads, wl.ctx, wl.head_dim), generator=g,
                                              device="cuda").to(torch.bfloat16)
    return kv


def make_engine(amk, wl, dev, opts):
    cfg = amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                          wl.vocab, wl.max_seq, wl.batch, wl.rms_eps, wl.rope_theta,
                          int8=wl.weight_dtype == "int8", tied=wl.tied,
                          int4=wl.weight_dtype == "int4", group_size=wl.group_size)
    return amk.DecodeEngine(cfg, dev["embed"], dev["final_norm"], dev["layers"], dev["lm_head"], dev["s_lm"],
                            opts or None)


class Timed:
    """One device-timed run of `steps` decode steps (one launch each) after
    `warmup` untimed ones, inputs resident in HBM.  The positions walk the
    workload's decode window from its context length and wrap around it."""

    def __init__(self, amk, eng, wl, kv, steps, warmup, local, dist=None):
        import numpy as np
        import torch
        B, window = wl.batch, wl.steps
        self.wl, self.steps, self.window = wl, steps, window
        stream = torch.cuda.current_stream()
        rng = np.random.default_rng(3)
        self.tok_host = rng.integers(0, wl.vocab, size=(window, B)).astype(np.int32)
        self.pos_host = np.ascontiguousarray((wl.ctx + np.arange(window, dtype=np.int32))[:, None].repeat(B, axis=1))
        tok_dev = torch.from_numpy(self.tok_host).cuda()
        pos_dev = torch.from_numpy(self.pos_host).cuda()
        self.logits = torch.empty((B, wl.vocab), dtype=torch.float32, device="cuda")
        h, lib, s_ptr = eng.handle, amk.lib(), stream.cuda_stream

        def launch(i):
            j = i % window
            st = lib.amk_decode_step(h, B, tok_dev[j].data_ptr(), pos_dev[j].data_ptr(), kv.data_ptr(),
                                     self.logits.data_ptr(), s_ptr)
            if st != amk.OK:
                raise amk.AmkError(st, "amk_decode_step")

        for i in range(warmup):
            launch(i)
        st = eng.sync()
        if st != amk.OK:
            raise amk.AmkError(st, "warm-up: %s" % eng.last_error())
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = NvmlClockSampler(local)
        if not sampler.ok:
            sampler = ClockSampler(local)
        with sampler as clocks:
            ev0.record(stream)
            for i in range(steps):
                launch(i)
            ev1.record(stream)
            torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        st = eng.sync()
        if st != amk.OK:
            raise amk.AmkError(st, "timed region: %s" % eng.last_error())
        self.ms = max_over_ranks(ms, dist, "cuda")
        self.ms_per_step = self.ms / steps
        self.clocks = clocks.summary()

    def roofline(self, traffic):
        wl, B = self.wl, self.wl.batch
        positions = [wl.ctx + (i % self.window) for i in range(self.steps)]
        alg = statistics.fmean(step_bytes(wl, p, B) for p in positions)
        peak, src = measured_peak()
        achieved = alg / (self.ms_per_step / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_source": src, "algorithmic_bytes_per_launch": alg,
                "frac_of_8TBps": achieved / NOMINAL_HBM_GBS, "kernel": "amk_decode_kernel"}


SUB_WORKLOADS = ("tinyllama_1b1_w8a16", "tinyllama_1b1_w4a16", "llama2_7b", "llama2_7b_b8", "smollm2_135m",
                 # the batch-size sweep on the short-sequence shape (64 prompt positions, 12 steps)
                 "tinyllama_1b1_short@1", "tinyllama_1b1_short@2", "tinyllama_1b1_short@4",
                 "tinyllama_1b1_short@8", "tinyllama_1b1_short@16",
                 # the same step as one launch per operator, CUDA-graphed
                 "unfused:tinyllama_1b1", "unfused:llama2_7b")


def unfused_record(amk, wl, steps, local):
    """The per-operator path (one launch per operator) on the same shape and
    device-filled data: one step captured in a CUDA graph, replayed `steps`
    times after warm-up, timed with CUDA events."""
    import numpy as np
    import torch
    dev = device_model(wl, seed=1)
    kv = device_kv(wl, seed=2, batch=wl.batch)
    cfg = amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                          wl.vocab, wl.max_seq, wl.batch, wl.rms_eps, wl.rope_theta,
                          int8=wl.weight_dtype == "int8", tied=wl.tied,
                          int4=wl.weight_dtype == "int4", group_size=wl.group_size)
    u = amk.UnfusedEngine(cfg, dev["embed"], dev["final_norm"], dev["layers"], dev["lm_head"], dev["s_lm"])
    tok = torch.ones(wl.batch, dtype=torch.int32, device="cuda")
    pos = torch.full((wl.batch,), wl.ctx, dtype=torch.int32, device="cuda")
    lg = torch.empty((wl.batch, wl.vocab), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            u.step(tok, pos, kv, lg, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        u.step(tok, pos, kv, lg, stream=s)
    for _ in range(8):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = NvmlClockSampler(local)
    if not sampler.ok:
        sampler = ClockSampler(local)
    with sampler as clocks:
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    u.close()
    n_launch = 3 + 13 * wl.n_layers
    return {"ms_per_step": ms, "us_per_token": 1e3 * ms / wl.batch, "tokens_per_s": wl.batch / (ms / 1e3),
            "steps": steps, "launches_per_step": n_launch, "clocks": clocks.summary(), "config": config_block(wl),
            "data": "synthetic, weights and KV filled on the device by torch's seeded generator",
            "what": "one kernel launch per operator, one step captured in a CUDA graph and replayed"}


def sub_records(amk, args, local):
    """The other targeted shapes on the same kernel, a few seconds each, with
    device-filled weights (device_model): 'name' is a workload, 'name@B' the
    workload at batch B, 'unfused:name' the per-operator path on it."""
    import synth
    import torch
    out = {}
    for name in args.sub:
        if name.startswith("unfused:"):
            out[name] = unfused_record(amk, synth.workload(name.split(":", 1)[1]), 64, local)
            torch.cuda.empty_cache()
            continue
        if "@" in name:
            base, b = name.split("@")
            wl = synth.workload(base, batch=int(b))
        else:
            wl = synth.workload(name)
        dev = device_model(wl, seed=1)
        kv = device_kv(wl, seed=2, batch=wl.batch)
        eng = make_engine(amk, wl, dev, None)
        steps = max(16, min(args.sub_steps, int(0.5e6 / max(1.0, 50.0 * wl.n_layers * wl.batch))))
        t = Timed(amk, eng, wl, kv, steps=steps, warmup=8, local=local)
        plan = eng.plan_info()
        out[name] = {"ms_per_step": t.ms_per_step, "us_per_token": 1e3 * t.ms_per_step / wl.batch,
                     "tokens_per_s": wl.batch / (t.ms_per_step / 1e3), "steps": steps, "warmup": 8,
                     "dtype": workload_dtype(wl), "config": config_block(wl), "clocks": t.clocks,
                     "roofline": t.roofline(traffic_from_profile(wl.name)),
                     "data": "synthetic, weights and KV filled on the device by torch's seeded generator",
                     "schedule": {k: plan[k] for k in ("att_chunks", "slot_bytes", "n_slots", "ksplit")}}
        eng.close()
        del dev, kv, eng
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2560)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="amk", choices=["amk", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sub", default=",".join(SUB_WORKLOADS),
                    help="comma-separated workloads timed as sub-records beside the headline ('' for none)")
    ap.add_argument("--sub-steps", type=int, default=512)
    ap.add_argument("--option", action="append", default=[], help="schedule option key=value (offline tuning)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.sub = [x for x in args.sub.split(",") if x]

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import synth
    # 'name@B' runs the workload at batch B (the batch sweep's shapes)
    name, _, bs = args.workload.partition("@")
    wl = synth.workload(name, **({"batch": int(bs)} if bs else {}))

    if args.impl == "reference":
        return reference_arm(args, wl, rank, world)

    import numpy as np
    import torch
    import persistent_sm_decode_gb300 as amk
    from synth.device import kv_to_device, model_to_device

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    amk.build()
    model = synth.make_model(wl, seed=1)
    kc, vc = synth.make_kv(wl, seed=2)
    dev = model_to_device(model)
    kv = kv_to_device(kc, vc)
    opts = {}
    for kvp in args.option:
        k, v = kvp.split("=")
        opts[k] = int(v)
    eng = make_engine(amk, wl, dev, opts)
    B = wl.batch
    stream = torch.cuda.current_stream()

    # ---- device-timed region: inputs resident, one launch per step ----
    t = Timed(amk, eng, wl, kv, args.steps, args.warmup, local, dist)
    value = whole_job_rate(world, B, args.steps, t.ms / 1e3)
    roofline = t.roofline(traffic_from_profile(wl.name))

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        window = wl.steps
        tok_pin = torch.from_numpy(t.tok_host).pin_memory()
        pos_pin = torch.from_numpy(t.pos_host).pin_memory()
        out_pin = torch.empty((B, wl.vocab), dtype=torch.float32).pin_memory()
        t_in = torch.empty((B,), dtype=torch.int32, device="cuda")
        p_in = torch.empty((B,), dtype=torch.int32, device="cuda")
        logits = t.logits
        n_e2e = min(args.steps, 512)
        for i in range(8):
            t_in.copy_(tok_pin[i % window], non_blocking=True)
            p_in.copy_(pos_pin[i % window], non_blocking=True)
            eng.step(t_in, p_in, kv, logits, stream=stream)
            out_pin.copy_(logits, non_blocking=True)
            stream.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            t_in.copy_(tok_pin[i % window], non_blocking=True)
            p_in.copy_(pos_pin[i % window], non_blocking=True)
            eng.step(t_in, p_in, kv, logits, stream=stream)
            out_pin.copy_(logits, non_blocking=True)
            stream.synchronize()   # the host needs the logits before it can pick the next token
        dt = max_over_ranks(time.perf_counter() - t0, dist, "cuda")
        e2e = {"value": whole_job_rate(world, B, n_e2e, dt), "unit": "tokens/s", "h2d_bytes_per_step": 2 * B * 4,
               "d2h_bytes_per_step": B * wl.vocab * 4, "steps": n_e2e, "us_per_token": 1e6 * dt / (B * n_e2e)}
        assert eng.sync() == amk.OK

    plan = eng.plan_info()
    eng.close()
    del dev, kv
    torch.cuda.empty_cache()

    subs = sub_records(amk, args, local) if (rank == 0 and world == 1 and args.sub) else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, n, threads, dt = time_oracle(model, kc, vc, wl, budget_s=15.0, max_steps=10 ** 6)
        tps1, n1, _, dt1 = time_oracle(model, kc, vc, wl, budget_s=5.0, max_steps=10 ** 6, threads=1)
        cpu = {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "%d decode steps of %s (%.1f s) on %s" % (n, wl.name, dt, cpu_model()),
               "us_per_token": 1e6 / tps,
               "single_thread": {"value": tps1, "unit": "tokens/s", "us_per_token": 1e6 / tps1,
                                 "sample": "%d decode steps (%.1f s) on one core" % (n1, dt1)}}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t.ms_per_step, "us_per_token": 1e3 * t.ms_per_step / B,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": workload_dtype(wl),
                "data": "synthetic", "config": config_block(wl),
                "clocks": t.clocks, "e2e": e2e, "gpu_launches": args.steps,
                "roofline": roofline, "cpu_baseline": cpu,
                "schedule": {k: plan[k] for k in ("n_sm", "att_chunks", "slot_bytes", "n_slots", "ksplit",
                                                  "scratch_depth", "smem_bytes", "n_tasks")},
                "kernel_sha": kernel_hash(), "workloads": subs}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
