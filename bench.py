"""Benchmark of the prompt-deduplication hot path on one GB300 (or N replicas).

One step = the whole path on one synthetic batch: find prompt groups, pack ids,
positions and the [B, L, 1024] hidden states, split attention forward and
backward on the packed Q/K/V/dO, and reconstruct the attention output back to
[B, L, Hq*D].  The headline value is useful split-attention fwd+bwd TFLOP/s
(attended pairs only) over the whole step, on the long-context workload (4
prompts of 32768 tokens x 8 responses of 2048, the largest configuration);
unique tokens per second, pack/reconstruct GB/s, the per-kernel roofline and
the same figures for every other configuration are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from dummy_batch import WORKLOADS, make_workload_batch, make_qkv, make_rows, bf16_round  # noqa: E402

METRIC = "split-attn fwd+bwd useful TFLOP/s (% BF16 peak); pack/reconstruct GB/s"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long_context"
# the other configurations, measured in the same run and reported by name
# (workload, use_unpad)
EXTRA_WORKLOADS = [("worked_example", False), ("qwen3_0p6b", False), ("pipeline", False),
                   ("pipeline", True), ("pipeline_nodedup", False)]
HIDDEN = 1024  # Qwen3-0.6B hidden size: the row width packed in every step

# Algorithmic FLOPs of the attention kernels per attended (query, key) pair,
# per query head and per unit of head_dim: a GEMM over the pairs costs 2 D.
KERNEL_FLOPS_PER_PAIR = {
    "attn_fwd": 4,    # S = Q K^T, O = P V
    "attn_dkdv": 8,   # S^T, dP^T, dV += P^T dO, dK += dS^T Q
    "attn_dq": 2,     # dQ += dS K (S and dP recomputed there are not counted)
    "attn_bwd": 10,   # the fused backward: S^T, dP^T, dV, dK and dQ
}
KERNEL_NAMES = {
    "attn_fwd": "attn_fwd_tc_kernel (split-attention forward)",
    "attn_dkdv": "attn_dkdv_tc_kernel (split-attention backward, dK and dV)",
    "attn_dq": "attn_dq_tc_kernel (split-attention backward, dQ)",
    "attn_bwd": "attn_bwd_tc_kernel (split-attention backward, dK, dV and dQ)",
}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--unpad", action="store_true", help="pack with use_unpad (needs a mask)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-standard", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other configurations")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args(argv)


def workload_desc(wl, use_unpad=False):
    resp = f"{wl.R}" if wl.resp_len_range is None else \
        f"{wl.resp_len_range[0]}..{wl.resp_len_range[1]} right-padded to {wl.R}"
    return (f"{wl.name}{' (unpadded)' if use_unpad else ''}: {wl.G} unique prompt(s) x {wl.n} responses "
            f"(B={wl.B}), prompt {wl.P}, response {resp}; {wl.Hq} Q / {wl.Hkv} KV heads, head_dim {wl.D}, "
            f"{wl.dtype}; {'forward + backward' if wl.backward else 'forward only'}; hidden {HIDDEN} packed")


def useful_pairs(info):
    """Attended (query, key) pairs of one head, from the reconstruction info
    arrays (split attention: prompt causal once, each response over prompt +
    own causal prefix)."""
    pairs = 0
    G = info["num_groups"]
    ptr = info["group_ptr"]
    for g in range(G):
        P = int(info["prompt_len"][g])
        pairs += P * (P + 1) // 2
        for i in range(ptr[g], ptr[g + 1]):
            m = int(info["resp_len"][info["members"][i]])
            pairs += m * P + m * (m + 1) // 2
    return pairs


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self):
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
               "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
               "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
               "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "50"]
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            cmd.insert(1, f"--id={vis.split(',')[int(os.environ.get('LOCAL_RANK', '0'))]}")
        else:
            cmd.insert(1, f"--id={int(os.environ.get('LOCAL_RANK', '0'))}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.samples.append([x.strip() for x in line.split(",")])
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        # nvidia-smi takes a moment to start: wait for its first sample so the
        # timed region is covered from its beginning
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.01)

    def mark(self):
        return len(self.samples)

    def stop(self, begin=0, end=None):
        """Summarise the samples taken between two mark() calls (plus the one
        in flight at the end); all samples if that window caught none."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = self.samples[begin:None if end is None else end + 1] or self.samples
        for s in window:
            try:
                sm.append(float(s[1]))
                mx = float(s[2])
                power.append(float(s[3]))
                for i, n in enumerate(names):
                    if s[5 + i].lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "power_w_median": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def kernel_source_digest(entry) -> str | None:
    """sha256 (16 hex digits) of what the traffic counters depend on: the
    source range of the kernel (from its config struct to the end of the
    kernel function) and the headers it includes."""
    import hashlib
    h = hashlib.sha256()
    try:
        text = open(os.path.join(ROOT, entry["source"])).read()
        a = text.index(entry["range_begin"])
        e = text.index(entry["range_end"], a)
        b = text.index("\n}\n", e) + 3
        h.update(text[a:b].encode())
        for dep in entry.get("headers", []):
            h.update(open(os.path.join(ROOT, dep), "rb").read())
    except (OSError, ValueError, KeyError):
        return None
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None when the kernel's source changed
    since the counters were taken.  A capture taken on a smaller case of the
    same kernel is scaled by the entry's stated factor for this workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None, None
    e = t.get(kernel)
    if not e or kernel_source_digest(e) != e.get("kernel_sha256_16"):
        return None, None
    if e.get("workload") == workload:
        return e.get("bytes_per_launch"), f"ncu capture on {workload}"
    factor = e.get("scale_to", {}).get(workload)
    if factor is None:
        return None, None
    return e["bytes_per_launch"] * factor, f"ncu capture on {e['workload']}, x{factor} ({e.get('scale_reason', '')})"


# ------------------------------------------------------- oracle (CPU arm)
class OracleSample:
    """The oracle as it stands, on a bounded sample of a workload: its batch,
    packing and seeded Q/K/V/dO are prepared once; each timed sample draws
    query rows uniformly from the packed batch and runs each row's split
    attention forward and its exact backward (sparse upstream gradient),
    every head."""

    def __init__(self, wl, use_unpad=False):
        import oracle
        self.oracle, self.wl = oracle, wl
        ids, mask, pos = make_workload_batch(wl, list(WORKLOADS).index(wl.name))
        groups, uniq = oracle.find_prompt_groups(ids, wl.R, mask)
        _, _, self.info = oracle.create_deduplicated_batch(ids, pos, wl.R, groups, uniq, attention_mask=mask,
                                                           use_unpad=use_unpad)
        self.q, self.k, self.v, self.do = make_qkv(self.info.T, wl.Hq, wl.Hkv, wl.D, 7)
        self.keysets = oracle.row_key_sets(self.info)
        self.valid_rows = np.flatnonzero(self.info.row_valid)
        self.rng = np.random.default_rng(0)
        self.per_row = (4.0 + 10.0) if wl.backward else 4.0
        self.cores = os.cpu_count()

    def run(self, seconds):
        """TFLOP/s of useful work over about `seconds` of sampled rows, and a
        description of the sample."""
        wl, oracle = self.wl, self.oracle
        flops = 0.0
        rows_done = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            rows = [int(self.valid_rows[int(i)]) for i in self.rng.integers(0, len(self.valid_rows), size=4)]
            oracle.split_attention_fwd_rows(self.q, self.k, self.v, self.info, rows, key_sets=self.keysets)
            if wl.backward:
                oracle.split_attention_bwd_sparse(self.q, self.k, self.v, self.do, self.info, rows,
                                                  key_sets=self.keysets)
            flops += sum(len(self.keysets[r]) for r in rows) * self.per_row * wl.D * wl.Hq
            rows_done += len(rows)
        el = time.perf_counter() - t0
        return flops / el / 1e12, (f"oracle (fp64 NumPy) split attention "
                                   f"{'fwd + exact bwd' if wl.backward else 'fwd'} on {rows_done} uniformly drawn "
                                   f"query rows x {wl.Hq} heads of the {wl.name} batch, {el:.1f} s; {self.cores} "
                                   f"host cores available to NumPy's BLAS")


def cpu_baseline(wl, seconds, use_unpad=False):
    """One bounded oracle sample of the workload: (TFLOP/s, cores, description)."""
    o = OracleSample(wl, use_unpad)
    v, desc = o.run(seconds)
    return v, o.cores, desc


def oracle_copy_times(wl, use_unpad=False, cols=64):
    """The oracle's grouping and packing of ids and positions, timed on the full
    batch; its row pack of the hidden states and its reconstruction of the
    attention output, timed on the full row set at `cols` float32 columns and
    scaled by width to the real rows (HIDDEN and Hq*D columns).  Seconds."""
    import oracle
    ids, mask, pos = make_workload_batch(wl, list(WORKLOADS).index(wl.name))
    t0 = time.perf_counter()
    groups, uniq = oracle.find_prompt_groups(ids, wl.R, mask)
    t1 = time.perf_counter()
    _, _, info = oracle.create_deduplicated_batch(ids, pos, wl.R, groups, uniq, attention_mask=mask,
                                                  use_unpad=use_unpad)
    t2 = time.perf_counter()
    rows = np.zeros((wl.B, wl.L, cols), dtype=np.float32)
    oracle.pack_rows(rows, info)
    t3 = time.perf_counter()
    oracle.reconstruct_sequences(np.zeros((info.T, cols), dtype=np.float32), info)
    t4 = time.perf_counter()
    return {"group_s": t1 - t0, "pack_ids_positions_s": t2 - t1,
            "pack_hidden_s_extrapolated": (t3 - t2) * HIDDEN / cols,
            "reconstruct_s_extrapolated": (t4 - t3) * (wl.Hq * wl.D) / cols,
            "note": f"group and ids/positions pack timed in full; hidden pack and reconstruction timed on "
                    f"every row at {cols} float32 columns and scaled by width to {HIDDEN} and {wl.Hq * wl.D} "
                    f"columns (extrapolated)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    use_unpad = bool(getattr(args, "unpad", False))
    per = max(args.cpu_seconds / max(args.steps + args.warmup, 1), 0.5)
    sample = OracleSample(wl, use_unpad)
    vals = []
    desc = None
    for i in range(args.warmup + args.steps):
        v, desc = sample.run(per)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    cores = sample.cores
    # the oracle's time for one whole step, extrapolated: the attention's useful
    # FLOPs at the sampled rate, plus the copy steps (timed, or scaled by width)
    import oracle
    info = sample.info
    pairs = oracle.attended_pairs([int(info.prompt_len[g]) for g in range(info.G)],
                                  [[int(info.resp_len[b]) for b in grp] for grp in info.prompt_groups])
    attn_flops = ((4.0 + 10.0) if wl.backward else 4.0) * wl.D * wl.Hq * pairs
    copies = oracle_copy_times(wl, use_unpad)
    attn_s = attn_flops / (value * 1e12)
    step_s = attn_s + copies["group_s"] + copies["pack_ids_positions_s"] + \
        copies["pack_hidden_s_extrapolated"] + copies["reconstruct_s_extrapolated"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "ms_per_step_kind": "extrapolated (see oracle_step)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(wl, use_unpad)},
            "oracle_step": {"attention_s_extrapolated": attn_s, "attention_flops": attn_flops,
                            "useful_pairs_per_head": pairs, "sample_seconds_per_step": per, **copies},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------ GPU arm
def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (every rank calls this; a no-op at N = 1).
    Throughput is then the units all ranks processed over that time."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


PHASES = ("group", "pack", "pack_hidden", "fwd", "bwd", "recon")


class Case:
    """One configuration on the device: its batch, persistent buffers and the
    whole-path step through the public binding."""

    def __init__(self, zr, wl, dev, use_unpad=False):
        import torch
        self.zr, self.wl, self.dev, self.use_unpad = zr, wl, dev, use_unpad
        idx = list(WORKLOADS).index(wl.name)
        self.ids_np, self.mask_np, self.pos_np = make_workload_batch(wl, idx)
        R = wl.R
        t_ids = torch.from_numpy(self.ids_np).to(dev)
        t_mask = None if self.mask_np is None else torch.from_numpy(self.mask_np).to(dev)
        t_pos = torch.from_numpy(self.pos_np).to(dev)
        self.t_ids, self.t_mask, self.t_pos = t_ids, t_mask, t_pos
        gen = torch.Generator(device=dev)
        gen.manual_seed(500 + idx)
        self.t_hidden = torch.randn((wl.B, wl.L, HIDDEN), generator=gen, device=dev, dtype=torch.float32).to(
            torch.bfloat16)
        # T from one untimed pass (sizes the packed buffers exactly)
        g = zr.find_prompt_groups(t_ids, R, t_mask, sync=True)
        _, _, _, info0, T = zr.pack_dedup(t_ids, t_pos, R, g, t_mask, use_unpad=use_unpad, sync=True)
        arrays = info0.arrays()
        self.G = arrays["num_groups"]
        self.pairs = useful_pairs(arrays)
        self.T = T
        self.fwd_flops = 4.0 * wl.D * wl.Hq * self.pairs
        self.bwd_flops = 10.0 * wl.D * wl.Hq * self.pairs if wl.backward else 0.0
        self.attn_flops = self.fwd_flops + self.bwd_flops
        T_cap = T
        self.T_cap = T_cap
        gen.manual_seed(900 + idx)
        self.tq, self.tk, self.tv, self.tdo = (
            torch.randn((T_cap, h, wl.D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            for h in (wl.Hq, wl.Hkv, wl.Hkv, wl.Hq))
        self.groups = zr.Groups(wl.B, dev)
        self.groups.unique_prompts = torch.empty((wl.B, wl.P), dtype=torch.int64, device=dev)
        self.grp_ws = zr._aligned_empty(zr.lib().zr_find_prompt_groups_workspace(wl.B, wl.L), dev)
        self.info = zr.ReconInfo(wl.B, wl.L, R, use_unpad, T_cap, dev)
        self.ids_out = torch.empty(T_cap, dtype=torch.int64, device=dev)
        self.pos_out = torch.empty(T_cap, dtype=torch.int64, device=dev)
        self.hid_out = torch.empty((T_cap, HIDDEN), dtype=torch.bfloat16, device=dev)
        self.attn_ws = zr.attn_workspace(self.info, wl.Hq, wl.Hkv, wl.D, dev)
        self.o = torch.empty_like(self.tq)
        self.lse = torch.empty((T_cap, wl.Hq), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(self.tq), torch.empty_like(self.tk), torch.empty_like(self.tv)
        self.recon = torch.empty((wl.B, wl.L, wl.Hq * wl.D), dtype=torch.bfloat16, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, ev=None, inputs=None, outputs=None):
        """The whole path once.  `ev` maps phase -> (start, end) events;
        `inputs` / `outputs` replace the resident tensors (end-to-end run)."""
        zr, wl = self.zr, self.wl
        ids, pos, mask, hidden, q, k, v, do = inputs or (self.t_ids, self.t_pos, self.t_mask, self.t_hidden,
                                                         self.tq, self.tk, self.tv, self.tdo)
        dq, dk, dv, recon = outputs or (self.dq, self.dk, self.dv, self.recon)

        def mark(name, i):
            if ev is not None:
                ev[name][i].record(self.stream)
        mark("group", 0)
        zr.find_prompt_groups(ids, wl.R, mask, workspace=self.grp_ws, out=self.groups)
        mark("group", 1)
        mark("pack", 0)
        zr.pack_dedup(ids, pos, wl.R, self.groups, mask, use_unpad=self.use_unpad, info=self.info,
                      out=(self.ids_out, self.pos_out, None))
        mark("pack", 1)
        mark("pack_hidden", 0)
        zr.pack_rows(self.info, hidden, out=self.hid_out)
        mark("pack_hidden", 1)
        mark("fwd", 0)
        zr.split_attn_fwd(self.info, q, k, v, workspace=self.attn_ws, out=(self.o, self.lse))
        mark("fwd", 1)
        mark("bwd", 0)
        if wl.backward:
            zr.split_attn_bwd(self.info, q, k, v, self.o, self.lse, do, workspace=self.attn_ws, out=(dq, dk, dv))
        mark("bwd", 1)
        mark("recon", 0)
        zr.reconstruct(self.info, self.o.view(self.T_cap, wl.Hq * wl.D), out=recon)
        mark("recon", 1)

    def measure(self, steps, warmup, flush, on_start=None):
        """Median phase times and the mean whole-step time (ms) over `steps`
        timed steps after `warmup` untimed ones; L2 flushed before every step,
        outside the timed events."""
        import torch
        ev = {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in PHASES}
        for _ in range(warmup):
            flush.zero_()
            self.step()
        torch.cuda.synchronize()
        self.zr.check_status(self.info, self.attn_ws)
        if on_start:
            on_start()
        times = {n: [] for n in PHASES}
        total = []
        for _ in range(steps):
            flush.zero_()
            self.step(ev)
            torch.cuda.synchronize()
            for n, (a, b) in ev.items():
                times[n].append(a.elapsed_time(b))
            total.append(ev["group"][0].elapsed_time(ev["recon"][1]))
        torch.cuda.synchronize()
        self.zr.check_status(self.info, self.attn_ws)
        return {n: statistics.median(v) for n, v in times.items()}, sum(total) / len(total)

    def summary(self, med, ms_step, peaks, world=1):
        """Throughput figures of one configuration."""
        wl = self.wl
        out = {"workload": workload_desc(wl, self.use_unpad), "B": wl.B, "L": wl.L, "T_packed": self.T,
               "groups": self.G, "useful_pairs_per_head": self.pairs, "ms_per_step": ms_step,
               "tflops_per_step": world * self.attn_flops / (ms_step * 1e-3) / 1e12,
               "unique_tokens_per_s": world * self.T / (ms_step * 1e-3),
               "batch_tokens_per_s": world * wl.B * wl.L / (ms_step * 1e-3),
               "breakdown_ms": med}
        out["frac_of_sustained_peak"] = out["tflops_per_step"] / (world * peaks["bf16_tflops_sustained"])
        out["attn_fwd_tflops"] = self.fwd_flops / (med["fwd"] * 1e-3) / 1e12
        if wl.backward:
            out["attn_bwd_tflops"] = self.bwd_flops / (med["bwd"] * 1e-3) / 1e12
        pack_bytes = 2 * self.T * HIDDEN * 2  # hidden rows: read once, written once
        recon_bytes = (self.T + wl.B * wl.L) * wl.Hq * wl.D * 2
        out["pack_hidden"] = {"bytes": pack_bytes, "gbs": pack_bytes / (med["pack_hidden"] * 1e-3) / 1e9}
        out["pack_hidden"]["frac_of_measured_hbm"] = out["pack_hidden"]["gbs"] / peaks["hbm_gbs"]
        out["reconstruct"] = {"bytes": recon_bytes, "gbs": recon_bytes / (med["recon"] * 1e-3) / 1e9}
        out["reconstruct"]["frac_of_measured_hbm"] = out["reconstruct"]["gbs"] / peaks["hbm_gbs"]
        return out


def run_native(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from prompt_deduplicated_shared_gb300 import zr

    peaks = load_peaks()
    wl = WORKLOADS[args.workload]
    # every rank processes its own batch (groups are independent units)
    case = Case(zr, wl, dev, use_unpad=args.unpad)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    clocks = ClockSampler()
    clocks.start()
    state = {}

    def on_start():
        zr.kernel_time_reset()
        zr.set_option("kernel_timing", 1)  # per-kernel event pairs, for the roofline
        state["launches0"] = zr.kernel_launches()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        state["clock_begin"] = clocks.mark()

    med, ms_local = case.measure(args.steps, args.warmup, flush, on_start=on_start)
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop(state["clock_begin"], clocks.mark())
    launches = zr.kernel_launches() - state["launches0"]
    zr.set_option("kernel_timing", 0)
    kernel_ms = {}
    for n in ("attn_fwd", "attn_bwd_prep", "attn_bwd", "attn_dkdv", "attn_dq", "attn_dq_convert",
              "pack_gather", "reconstruct"):
        tot, cnt = zr.kernel_time(n)
        if cnt:
            kernel_ms[n] = {"launches": cnt, "avg_ms": tot / cnt, "total_ms": tot}
    zr.kernel_time_reset()
    timed_total = sum(k["total_ms"] for k in kernel_ms.values())
    for k in kernel_ms.values():
        k["share_of_timed_kernels"] = k["total_ms"] / timed_total if timed_total else None

    ms_step = max_over_ranks(ms_local, world, dev)
    value = world * case.attn_flops / (ms_step * 1e-3) / 1e12
    summ = case.summary(med, ms_step, peaks, world)

    # dominant kernel: the attention kernel with the largest share of the timed
    # events; its algorithmic FLOPs per launch over its mean event time
    attn_k = [n for n in kernel_ms if n in KERNEL_FLOPS_PER_PAIR]
    dom = max(attn_k, key=lambda n: kernel_ms[n]["total_ms"])
    dom_flops = KERNEL_FLOPS_PER_PAIR[dom] * wl.D * wl.Hq * case.pairs
    dom_ms = kernel_ms[dom]["avg_ms"]
    dom_tflops = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic, traffic_src = load_traffic(dom, wl.name if not args.unpad else wl.name + "_unpad")
    kernel_tflops = {n: KERNEL_FLOPS_PER_PAIR[n] * wl.D * wl.Hq * case.pairs / (kernel_ms[n]["avg_ms"] * 1e-3) / 1e12
                     for n in attn_k}

    # the reconstruction adjoint (backward through the reconstruction of the
    # attention output), timed on its own: it is not one of the steps above
    grad_recon = torch.randn_like(case.recon)
    grad_packed = torch.empty((case.T_cap, wl.Hq * wl.D), dtype=torch.bfloat16, device=dev)
    rb_times = []
    for i in range(args.warmup + 10):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(case.stream)
        zr.reconstruct_backward(case.info, grad_recon, out=grad_packed)
        b.record(case.stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            rb_times.append(a.elapsed_time(b))
    zr.check_status(case.info, case.attn_ws)
    rb_ms = statistics.median(rb_times)
    rb_bytes = (wl.B * wl.L + case.T) * wl.Hq * wl.D * 2  # every output row read once, packed rows written
    rb_gbs = rb_bytes / (rb_ms * 1e-3) / 1e9
    del grad_recon, grad_packed

    # the standard strategy ("Split Attention Optimization", use_split_attention
    # off): reconstruct Q, K, V to the full sequences and run ordinary causal
    # attention on them (identity grouping); attention fwd + bwd only, timed
    # apart from the step as the in-repo baseline of the split path
    std = None
    if not args.no_standard:
        gi = zr.identity_groups(wl.B, dev)
        _, _, _, info_id, T_id = zr.pack_dedup(case.t_ids, case.t_pos, wl.R, gi, case.t_mask, sync=True)
        qf, kf, vf, dof = (zr.reconstruct(case.info, x.view(case.T_cap, -1)).view(wl.B * wl.L, x.shape[1], wl.D)
                           for x in (case.tq, case.tk, case.tv, case.tdo))
        ws_id = zr.attn_workspace(info_id, wl.Hq, wl.Hkv, wl.D, dev)
        of, lsef = torch.empty_like(qf), torch.empty((T_id, wl.Hq), dtype=torch.float32, device=dev)
        dqf, dkf, dvf = torch.empty_like(qf), torch.empty_like(kf), torch.empty_like(vf)
        st_times = []
        for i in range(4):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(case.stream)
            zr.split_attn_fwd(info_id, qf, kf, vf, workspace=ws_id, out=(of, lsef))
            if wl.backward:
                zr.split_attn_bwd(info_id, qf, kf, vf, of, lsef, dof, workspace=ws_id, out=(dqf, dkf, dvf))
            b.record(case.stream)
            torch.cuda.synchronize()
            if i > 0:
                st_times.append(a.elapsed_time(b))
        zr.check_status(info_id, ws_id)
        std_ms = statistics.median(st_times)
        split_ms = med["fwd"] + med["bwd"]
        std = {"ms_attention": std_ms, "split_ms_attention": split_ms, "speedup_of_split": std_ms / split_ms,
               "note": "same kernels on the reconstructed full sequences, every row its own group"}
        del qf, kf, vf, dof, of, lsef, dqf, dkf, dvf, ws_id
        torch.cuda.empty_cache()

    # end to end: host buffers in, results out, through the same public API.
    # Every step copies its inputs from pinned host memory and its results
    # (dQ, dK, dV and the reconstructed attention output) back to pinned host
    # memory; copies run on their own streams, double-buffered, so step i+1's
    # upload and step i-1's download overlap step i's kernels.
    e2e = None
    if not args.no_e2e:
        h_ids = torch.from_numpy(case.ids_np).pin_memory()
        h_pos = torch.from_numpy(case.pos_np).pin_memory()
        h_mask = None if case.mask_np is None else torch.from_numpy(case.mask_np).pin_memory()
        h_in = [h_ids, h_pos, h_mask] + [x.cpu().pin_memory() for x in
                                         (case.t_hidden, case.tq, case.tk, case.tv, case.tdo)]
        outs = [[torch.empty_like(x) for x in (case.dq, case.dk, case.dv, case.recon)] for _ in range(2)]
        h_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (case.dq, case.dk, case.dv, case.recon)]
                 for _ in range(2)]
        d_in = [[None if x is None else torch.empty(x.shape, dtype=x.dtype, device=dev) for x in h_in]
                for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in h_in if x is not None)
        d2h = sum(x.numel() * x.element_size() for x in h_out[0])
        s_up = torch.cuda.Stream(dev)
        s_down = torch.cuda.Stream(dev)
        ev_in_ready = [torch.cuda.Event() for _ in range(2)]
        ev_in_free = [torch.cuda.Event() for _ in range(2)]
        ev_out_ready = [torch.cuda.Event() for _ in range(2)]
        ev_out_free = [torch.cuda.Event() for _ in range(2)]
        for e in ev_in_free + ev_out_free:
            e.record(case.stream)

        def e2e_step(i):
            j = i & 1
            with torch.cuda.stream(s_up):
                s_up.wait_event(ev_in_free[j])
                for d, h in zip(d_in[j], h_in):
                    if h is not None:
                        d.copy_(h, non_blocking=True)
                ev_in_ready[j].record(s_up)
            case.stream.wait_event(ev_in_ready[j])
            case.stream.wait_event(ev_out_free[j])
            case.step(inputs=d_in[j], outputs=outs[j])
            ev_in_free[j].record(case.stream)
            ev_out_ready[j].record(case.stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_out_ready[j])
                for h, d in zip(h_out[j], outs[j]):
                    h.copy_(d, non_blocking=True)
                ev_out_free[j].record(s_down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(3, min(args.steps, 10))
        t_start.record(s_up)
        for i in range(n_e2e):
            e2e_step(i)
        t_end.record(s_down)
        torch.cuda.synchronize()
        zr.check_status(case.info, case.attn_ws)
        ms_e2e = max_over_ranks(t_start.elapsed_time(t_end) / n_e2e, world, dev)
        e2e = {"value": world * case.attn_flops / (ms_e2e * 1e-3) / 1e12, "unit": UNIT,
               "ms_per_step": ms_e2e, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "unique_tokens_per_s": world * case.T / (ms_e2e * 1e-3),
               "overlap": "uploads, kernels and downloads of consecutive steps overlap on separate streams"}
        del h_in, outs, h_out, d_in
    T_main = case.T
    del case
    torch.cuda.empty_cache()

    # the other configurations, each its own whole-path step
    extras = {}
    if not args.no_extras:
        for name, unpad in EXTRA_WORKLOADS:
            if name == wl.name and unpad == args.unpad:
                continue
            c = Case(zr, WORKLOADS[name], dev, use_unpad=unpad)
            m, ms = c.measure(max(5, min(args.steps, 10)), args.warmup, flush)
            ms = max_over_ranks(ms, world, dev)
            extras[name + ("_unpad" if unpad else "")] = c.summary(m, ms, peaks, world)
            del c
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, cores, desc = cpu_baseline(wl, args.cpu_seconds, args.unpad)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(wl, args.unpad), "B": wl.B, "L": wl.L, "T_packed": T_main,
                   "useful_pairs_per_head": summ["useful_pairs_per_head"], "fwd_flops": 4.0 * wl.D * wl.Hq * summ["useful_pairs_per_head"],
                   "bwd_flops": (10.0 if wl.backward else 0.0) * wl.D * wl.Hq * summ["useful_pairs_per_head"],
                   "l2": "flushed before every step (256 MiB write, outside the timed events); inputs exceed L2",
                   "parallelism": f"replicas x{world} (independent batches)"},
        "tokens_per_s": summ["unique_tokens_per_s"],
        "tokens_per_s_note": "unique (packed) tokens per second over the whole step; batch_tokens_per_s counts B*L",
        "batch_tokens_per_s": summ["batch_tokens_per_s"],
        "frac_of_sustained_peak": value / (world * peaks["bf16_tflops_sustained"]),
        "frac_of_burst_peak": value / (world * peaks["bf16_tflops"]),
        "roofline": {"kernel": KERNEL_NAMES[dom], "bound": "tensor", "achieved": dom_tflops,
                     "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": dom_tflops / peaks["bf16_tflops_sustained"],
                     "frac_of_burst": dom_tflops / peaks["bf16_tflops"],
                     "traffic": traffic, "traffic_source": traffic_src,
                     "flops_per_launch": dom_flops, "launch_ms": dom_ms,
                     "peak_source": f"{peaks['source']} bf16 dense, sustained (MEASURED_PEAKS.json): the kernel "
                                    f"runs inside a seconds-long loop of steps"},
        "kernels": kernel_ms,
        "kernel_tflops": kernel_tflops,
        "breakdown_ms": med,
        "attn_fwd": {"tflops": summ["attn_fwd_tflops"],
                     "frac_of_sustained_peak": summ["attn_fwd_tflops"] / peaks["bf16_tflops_sustained"]},
        "attn_bwd": None if not wl.backward else {
            "tflops": summ["attn_bwd_tflops"],
            "frac_of_sustained_peak": summ["attn_bwd_tflops"] / peaks["bf16_tflops_sustained"]},
        "pack": {"kernel": "pack_rows of the [B, L, 1024] bf16 hidden states", **summ["pack_hidden"],
                 "ids_positions_ms": med["pack"]},
        "reconstruct": {"kernel": "reconstruct of the attention output [T, Hq*D] bf16 to [B, L, Hq*D]",
                        **summ["reconstruct"]},
        "reconstruct_backward": {"kernel": "adjoint of the reconstruction, [B, L, Hq*D] bf16 gradient to [T, Hq*D] "
                                           "(shared prompt rows summed over members); timed apart from the step",
                                 "bytes": rb_bytes, "ms": rb_ms, "gbs": rb_gbs,
                                 "frac_of_measured_hbm": rb_gbs / peaks["hbm_gbs"]},
        "standard_attention": std,
        "workloads": extras,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
