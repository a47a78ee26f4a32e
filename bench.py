"""Benchmark of the affix-cache attention hot path on one GB300 (replicas for N > 1).

One step = one pass of the whole path over one batch of the LLaDA-8B-shaped prefix
workload (32 layers, 32 heads, head_dim 128, batch 4, affix L = 1024, 128 request +
256 masked rows, anchor ratio 0.2 -> K = 205, R = 589, 8 recompute points):
  anchor probe of all 32 layers (probe forward + masked-to-affix mass)  -> scores
  Top-K anchors -> admission maps
  8 recompute points x 32 layers x (anchor_write of R rows + slot attention R x T).

Prints ONE JSON line (rank 0).  Metric: probe + slot-attention TFLOP/s (algorithmic
flops: 4*P*T*d per probe row-head-layer, 4*R*T*d per recompute row-head-layer).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from affix_kv_cache_gb300 import workloads as wl  # noqa: E402

METRIC = "probe+slot_attn TFLOP/s & % of GB300 bf16 peak; anchor-scored tokens/s"
DEFAULT_WORKLOAD = wl.LLADA_PREFIX.name


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(wl.CATALOGUE))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="skip the block-decode measurement")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the compact per-launch record of the other workloads in the JSON line")
    ap.add_argument("--sweep", action="store_true",
                    help="per-launch measurements of the other workloads (Dream GQA infix, paged "
                         "LLaDA decode, long suffix with its ratio and batch sweeps), one JSON line each")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle sample")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run this many layers instead of the workload's")
    ap.add_argument("--points", type=int, default=0,
                    help="profiling only: recompute points per step instead of the workload's")
    ap.add_argument("--decode-only", action="store_true",
                    help="profiling only: one step to build the maps, then the block-decode "
                         "measurement alone (its JSON record)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- flops
def probe_flops(w, batch=None):
    return 4.0 * w.P * w.T * w.d * w.hq * w.layers * (batch or w.batch)


def slot_flops_per_launch(w, batch=None):
    return 4.0 * w.R * w.T * w.d * w.hq * (batch or w.batch)


def step_flops(w):
    return probe_flops(w) + slot_flops_per_launch(w) * w.layers * w.recompute_points


# ----------------------------------------------------------------------------- peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def profiled_traffic(kernel_files, workload, summary="slot_attention_llada8b_prefix.md"):
    """DRAM bytes per launch of a kernel from its committed ncu summary, or None if the
    summary is missing, was taken on another workload, or the kernel source changed since it
    was captured."""
    import hashlib
    summ = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(summ):
        return None
    fields = {}
    for line in open(summ):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    h = hashlib.sha256()
    for f in kernel_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if fields.get("source_sha256") != h.hexdigest()[:16] or fields.get("workload") != workload:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # nvidia-smi takes a moment to start: wait (up to 3 s) for its first sample, then count
        # only the samples taken from here on, inside the timed region
        self.skip = 0
        if self.proc is not None:
            t_end = time.time() + 3.0
            while time.time() < t_end and self.proc.poll() is None:
                self.f.flush()
                if os.path.exists(self.path) and os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.02)
            self.skip = sum(1 for _ in open(self.path)) if os.path.exists(self.path) else 0
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, device_index=0):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for n_line, line in enumerate(open(self.path)):
            if n_line < self.skip:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9 or not parts[0].isdigit() or int(parts[0]) != device_index:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        under = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(under) if under else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- the path
class Path:
    """Device-resident inputs of one workload plus the sequence of C-ABI calls of a step."""

    def __init__(self, w, device, seed_offset=0):
        import affix_kv_cache_gb300 as ac
        self.ac = ac
        self.w = w = w.replace(seed=w.seed + seed_offset)
        self.dev = device
        self.desc = ac.attn_desc(w.hq, w.hkv, w.d, w.scale, w.dtype)
        lay = wl.slot_layout(w, device)
        self.lay = lay
        self.masked = torch.tensor(w.masked_rows(), dtype=torch.int32, device=device).expand(
            w.batch, -1).contiguous()
        self.probe = [wl.probe_inputs(w, n, device) for n in range(w.layers)]
        self.rec = [wl.recompute_inputs(w, n, 0, device) for n in range(w.layers)]
        self.kc = [torch.zeros((lay.num_slots, w.hkv, w.d), dtype=w.torch_dtype, device=device)
                   for _ in range(w.layers)]
        self.vc = [torch.zeros_like(k) for k in self.kc]
        for n in range(w.layers):   # register the shared affix cache once (admission)
            ac.acache_write_slots(self.desc, 1, w.L, lay.shared_slot, self.probe[n]["k_aff"],
                                  self.probe[n]["v_aff"], self.kc[n], self.vc[n], lay.num_slots, 0)
        self.scores = torch.zeros((w.batch, w.L), dtype=torch.float32, device=device)
        self.ws_bytes = ac.acache_probe_workspace_bytes(self.desc, w.batch, w.T, w.L, w.m)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.probe_out = torch.empty_like(self.probe[0]["q"])
        self.anchors = torch.empty((w.batch, w.K), dtype=torch.int32, device=device)
        self.write_pos = torch.empty((w.batch, w.R), dtype=torch.int32, device=device)
        self.read_slot = torch.empty((w.batch, w.T), dtype=torch.int32, device=device)
        self.out = [torch.empty_like(r["q_r"]) for r in self.rec]
        self.k_new_l = [r["k_new"] for r in self.rec]
        self.v_new_l = [r["v_new"] for r in self.rec]
        self.q_r_l = [r["q_r"] for r in self.rec]
        self.launches_per_step = w.layers * 3 + 2 + w.recompute_points * w.layers * 2
        torch.cuda.synchronize()

    def probe_lists(self):
        """Per-layer q, k_req, v_req, k_aff, v_aff lists of the probe inputs in use."""
        return [[p[k] for p in self.probe] for k in ("q", "k_req", "v_req", "k_aff", "v_aff")]

    def step(self, ev=None):
        """One pass of the path.  `ev` (optional) collects CUDA events around phases."""
        ac, w, lay = self.ac, self.w, self.lay
        s = torch.cuda.current_stream()
        self.scores.zero_()
        if ev is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
        # the probe of every layer in one call (later layers' grids chained behind earlier ones)
        ac.acache_probe_scores_layers(self.desc, w.batch, w.T, w.l, w.L, self.masked, w.m,
                                      *self.probe_lists(), [self.probe_out] * w.layers, self.scores,
                                      self.ws, self.ws_bytes)
        if ev is not None:
            ep = torch.cuda.Event(enable_timing=True)
            ep.record(s)
            ev["probe"].append((e0, ep))
        ac.acache_topk_anchors(self.scores, w.batch, w.L, w.K, self.anchors)
        if ev is not None:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(s)
            ev["select"].append((e0, e1))
        ac.acache_build_slot_maps(w.batch, w.T, w.l, w.L, w.K, self.anchors, lay.shared_slot,
                                  lay.private_slots, self.write_pos, self.read_slot)
        for _ in range(w.recompute_points):
            # one recompute point over all layers in one call: the stores of every layer, then
            # the attentions, their grids chained
            ac.acache_store_attend_layers(self.desc, w.batch, w.R, lay.private_slots, self.k_new_l,
                                          self.v_new_l, self.kc, self.vc, lay.num_slots, lay.private_begin,
                                          w.R, self.q_r_l, w.T, self.read_slot, self.out)

    # ---- host buffers for the end-to-end measurement ---------------------------------
    UPLOADED = ("q", "k_req", "v_req")     # probe inputs a step takes from the host (the affix
                                          # K/V is the resident shared cache)

    def host_inputs(self):
        """Pinned host copies of every input a step takes from the host, and a second set of
        device input buffers: step k computes on set k % 2 while step k+1's inputs upload
        into the other set on a copy stream."""
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        self.h_probe = [{k: pin(p[k]) for k in self.UPLOADED} for p in self.probe]
        self.h_rec = [{k: pin(v) for k, v in r.items()} for r in self.rec]
        self.h_anchors = torch.empty(self.anchors.shape, dtype=torch.int32).pin_memory()
        self.h_scores = torch.empty(self.scores.shape, dtype=torch.float32).pin_memory()
        self.h_out = torch.empty(self.out[-1].shape, dtype=self.out[-1].dtype).pin_memory()
        bi = sum(t.numel() * t.element_size() for p in self.h_probe for t in p.values())
        bi += sum(t.numel() * t.element_size() for r in self.h_rec for t in r.values())
        bo = sum(t.numel() * t.element_size() for t in (self.h_anchors, self.h_scores, self.h_out))
        second_probe = [dict(p, **{k: torch.empty_like(p[k]) for k in self.UPLOADED}) for p in self.probe]
        second_rec = [{k: torch.empty_like(v) for k, v in r.items()} for r in self.rec]
        self.sets = [(self.probe, self.rec), (second_probe, second_rec)]
        self.copy_stream = torch.cuda.Stream()
        self.ev_ready = [torch.cuda.Event(), torch.cuda.Event()]   # a set's inputs are uploaded
        self.ev_used = [torch.cuda.Event(), torch.cuda.Event()]    # a set's step is done with them
        for e in self.ev_used:
            e.record()
        return bi, bo

    def use_set(self, i):
        self.probe, self.rec = self.sets[i]
        self.k_new_l = [r["k_new"] for r in self.rec]
        self.v_new_l = [r["v_new"] for r in self.rec]
        self.q_r_l = [r["q_r"] for r in self.rec]

    def upload(self, i):
        """Copy a step's inputs from pinned host memory into device set i (copy stream), once
        the step that last used set i is done with it."""
        cs = self.copy_stream
        cs.wait_event(self.ev_used[i])
        probe, rec = self.sets[i]
        with torch.cuda.stream(cs):
            for n in range(self.w.layers):
                for k, v in self.h_probe[n].items():
                    probe[n][k].copy_(v, non_blocking=True)
                for k, v in self.h_rec[n].items():
                    rec[n][k].copy_(v, non_blocking=True)
        self.ev_ready[i].record(cs)

    def step_e2e(self, k, upload_next=True):
        """Step k end to end: it waits for its inputs (uploaded into set k % 2), computes on
        them and reads its results back (scores, anchors, the last layer's attention output)
        into pinned host memory; meanwhile the next step's inputs upload into the other set."""
        s = torch.cuda.current_stream()
        cur = k % 2
        if upload_next:
            self.upload(1 - cur)
        s.wait_event(self.ev_ready[cur])
        self.use_set(cur)
        self.step()
        self.ev_used[cur].record(s)
        self.h_anchors.copy_(self.anchors, non_blocking=True)
        self.h_scores.copy_(self.scores, non_blocking=True)
        self.h_out.copy_(self.out[-1], non_blocking=True)

    def upload_ms(self, reps=3):
        """Milliseconds to upload one step's inputs with nothing else running: the host link's
        share of the end-to-end step (the link is shared with the machine's other GPUs)."""
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(self.copy_stream)
        for _ in range(reps):
            self.upload(0)
        z.record(self.copy_stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) / reps


class Decode:
    """Block-decode steps on a Path's pools: per layer, the current block's fresh K/V are
    written into the private slots of its positions, then its queries attend over all T
    logical keys through the read map (one write + one slot attention launch per layer)."""

    STEPS = 4   # distinct blocks cycled through

    def __init__(self, path):
        self.p = p = path
        w = p.w
        self.blocks = [wl.decode_block_positions(w, s) for s in range(self.STEPS)]
        self.n = len(self.blocks[0])
        self.inp = [[wl.decode_inputs(w, n, s, p.dev) for n in range(w.layers)] for s in range(self.STEPS)]
        self.wslot = [p.read_slot[:, torch.tensor(b, device=p.dev)].contiguous() for b in self.blocks]
        self.out = torch.empty_like(self.inp[0][0]["q_blk"])
        # bytes a launch must move at least once: every distinct slot the batch reads (K and
        # V), the queries, the output and the read map
        distinct = int(torch.unique(p.read_slot).numel())
        row = w.hkv * w.d * w.esize
        qo = 2 * w.batch * self.n * w.hq * w.d * w.esize
        self.unique_bytes = 2 * distinct * row + qo + w.batch * w.T * 4
        self.logical_bytes = 2 * w.batch * w.T * row + qo + w.batch * w.T * 4
        self.write_bytes = 2 * 2 * w.batch * self.n * row          # K and V, read + written

    def run(self, step, kinds=("write", "attn")):
        p, w, ac = self.p, self.p.w, self.p.ac
        i = step % self.STEPS
        for n in range(w.layers):
            d = self.inp[i][n]
            if "write" in kinds:
                ac.acache_write_slots(p.desc, w.batch, self.n, self.wslot[i], d["k_blk"], d["v_blk"],
                                      p.kc[n], p.vc[n], p.lay.num_slots, p.lay.private_begin)
            if "attn" in kinds:
                ac.acache_slot_attention(p.desc, w.batch, self.n, d["q_blk"], w.T, p.read_slot,
                                         p.kc[n], p.vc[n], p.lay.num_slots, self.out)
            if "fused" in kinds:
                ac.acache_store_attend(p.desc, w.batch, self.n, self.wslot[i], d["k_blk"], d["v_blk"],
                                       p.kc[n], p.vc[n], p.lay.num_slots, p.lay.private_begin, self.n,
                                       d["q_blk"], w.T, p.read_slot, self.out)

    def measure(self, reps, warmup, peaks):
        """Times CUDA-graph replays of STEPS blocks x all layers: the decode loop is
        launch-bound, so the launches are captured once and replayed without host work."""
        for k in range(warmup):
            self.run(k)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        graphs = {}
        for name, kinds in (("step", ("write", "attn")), ("attn", ("attn",)), ("write", ("write",)),
                            ("fused", ("fused",))):
            g = torch.cuda.CUDAGraph()
            try:
                with torch.cuda.graph(g, stream=side):
                    for i in range(self.STEPS):
                        self.run(i, kinds)
            except Exception as e:   # a capture the driver refuses is reported, not fatal
                graphs[name] = None
                print(f"decode: capture of {name} failed: {e}", file=sys.stderr)
                continue
            graphs[name] = g
        torch.cuda.synchronize()
        w = self.p.w
        per = self.STEPS * w.layers          # launches of each kind per replay

        def replay_ms(g):
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        t_step, t_attn, t_write = (replay_ms(graphs[k]) for k in ("step", "attn", "write"))
        t_fused = replay_ms(graphs["fused"]) if graphs.get("fused") is not None else None
        attn_ms, write_ms = t_attn / per, t_write / per
        achieved = self.unique_bytes / (attn_ms / 1e3) / 1e9
        # the kernel the library picks for this geometry (one query head per KV head and enough
        # requests: the recompute kernel, whose lone query tile splits the keys over two chains)
        path = self.p.ac.acache_slot_attention_path(self.p.desc, w.batch, self.n, w.T)
        kernel, src = {self.p.ac._lib.ACACHE_PATH_RECOMPUTE: ("tc_attn_kernel (split keys)", "tc_attn.cu"),
                       self.p.ac._lib.ACACHE_PATH_RECOMPUTE_PERSISTENT: ("tc_slot_persist_kernel (split keys)",
                                                                        "tc_attn.cu"),
                       self.p.ac._lib.ACACHE_PATH_BLOCK_DECODE: ("tc_decode_kernel", "tc_decode.cu")}.get(
                           path, ("simt", None))
        return {
            "workload": w.name, "block": self.n, "layers": w.layers, "replays": reps,
            "timing": f"CUDA graph replay, {per} launches of each kind per replay",
            "ms_per_layer": t_step / per, "attn_ms_per_launch": attn_ms, "write_ms_per_launch": write_ms,
            "store_attend_ms_per_layer": None if t_fused is None else t_fused / per,
            "attn_tflops": 4.0 * self.n * w.T * w.d * w.hq * w.batch / (attn_ms / 1e3) / 1e12,
            "logical_gather_gbs": self.logical_bytes / (attn_ms / 1e3) / 1e9,
            "write_gbs": self.write_bytes / (write_ms / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "peak_source": f"{peaks['source']} HBM copy",
                         "bytes_per_launch": self.unique_bytes,
                         "traffic": None if src is None else profiled_traffic(
                             [f"affix_kv_cache_gb300/csrc/{src}"], w.name, "decode_slot_attention_llada8b_prefix.md")},
        }


def slot_launch_times(path, reps=3):
    """The read-slot attention of one recompute point over all layers, timed two ways with
    CUDA events: chained as the step runs it (acache_store_attend_layers with no store, one
    call; ms per launch = the call / layers), and one launch at a time (events around each
    acache_slot_attention).  Returns (chained, alone) ms per launch."""
    ac, w, lay = path.ac, path.w, path.lay

    def chained():
        ac.acache_store_attend_layers(path.desc, w.batch, 0, None, None, None, path.kc, path.vc, lay.num_slots,
                                      lay.private_begin, w.R, path.q_r_l, w.T, path.read_slot, path.out)

    chained()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        chained()
    b.record()
    torch.cuda.synchronize()
    t_chain = a.elapsed_time(b) / (reps * w.layers)
    pairs = []
    for _ in range(reps):
        for n in range(w.layers):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ac.acache_slot_attention(path.desc, w.batch, w.R, path.q_r_l[n], w.T, path.read_slot, path.kc[n],
                                     path.vc[n], lay.num_slots, path.out[n])
            e1.record()
            pairs.append((e0, e1))
    torch.cuda.synchronize()
    t_alone = statistics.mean(e0.elapsed_time(e1) for e0, e1 in pairs)
    return t_chain, t_alone


def store_attend_compare(path, reps=3):
    """One recompute point over all layers: the store and the attention as two calls, against
    acache_store_attend (one call; the attention grid starts while the store drains).
    Returns ms per layer of each, from CUDA events around `reps` passes."""
    ac, w, lay = path.ac, path.w, path.lay

    def run(fused):
        for n in range(w.layers):
            r = path.rec[n]
            if fused:
                ac.acache_store_attend(path.desc, w.batch, w.R, lay.private_slots, r["k_new"], r["v_new"],
                                       path.kc[n], path.vc[n], lay.num_slots, lay.private_begin, w.R,
                                       r["q_r"], w.T, path.read_slot, path.out[n])
            else:
                ac.acache_write_slots(path.desc, w.batch, w.R, lay.private_slots, r["k_new"], r["v_new"],
                                      path.kc[n], path.vc[n], lay.num_slots, lay.private_begin)
                ac.acache_slot_attention(path.desc, w.batch, w.R, r["q_r"], w.T, path.read_slot,
                                         path.kc[n], path.vc[n], lay.num_slots, path.out[n])

    def run_layers():
        ac.acache_store_attend_layers(path.desc, w.batch, w.R, lay.private_slots, path.k_new_l, path.v_new_l,
                                      path.kc, path.vc, lay.num_slots, lay.private_begin, w.R, path.q_r_l, w.T,
                                      path.read_slot, path.out)

    res = {}
    for name, fused in (("separate_ms_per_layer", False), ("store_attend_ms_per_layer", True),
                        ("store_attend_layers_ms_per_layer", None)):
        fn = run_layers if fused is None else (lambda f=fused: run(f))
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        res[name] = a.elapsed_time(b) / (reps * w.layers)
    return res


def copy_bandwidth(path, peaks, reps=3):
    """The two HBM-bound copies alone, over every layer: the store (anchor_write of the R fresh
    rows per request) and the logical-KV gather through the read-slot map (acache_gather_slots,
    T rows per request).  Algorithmic bytes per launch = every row read once + written once,
    K and V; GB/s from CUDA events around `reps` passes."""
    ac, w, lay = path.ac, path.w, path.lay
    row = w.hkv * w.d * torch.tensor([], dtype=w.torch_dtype).element_size()
    k_out = torch.empty((w.batch, w.T, w.hkv, w.d), dtype=w.torch_dtype, device="cuda")
    v_out = torch.empty_like(k_out)

    def store():
        for n in range(w.layers):
            r = path.rec[n]
            ac.acache_write_slots(path.desc, w.batch, w.R, lay.private_slots, r["k_new"], r["v_new"],
                                  path.kc[n], path.vc[n], lay.num_slots, lay.private_begin)

    def gather():
        for n in range(w.layers):
            ac.acache_gather_slots(path.desc, w.batch, w.T, path.read_slot, path.kc[n], path.vc[n],
                                   lay.num_slots, k_out, v_out)

    res = {}
    for name, fn, rows in (("store", store, w.batch * w.R), ("gather", gather, w.batch * w.T)):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / (reps * w.layers)
        nbytes = 2 * 2 * rows * row                      # K and V, read once and written once
        gbs = nbytes / (ms / 1e3) / 1e9
        res[name] = {"ms_per_launch": ms, "bytes_per_launch": nbytes, "gbs": gbs,
                     "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} HBM copy"}
    return res


# ----------------------------------------------------------------------------- oracle
def cpu_oracle_sample(w, budget_s):
    """Time the oracle as it stands on a bounded sample of the workload: request 0, layer by
    layer, the probe of all heads and then the slot attention of a slice of the recomputed
    rows, until the budget is spent.  Returns (flops, seconds, cores, description)."""
    import numpy as np
    import oracle
    w1 = w.replace(batch=1)
    lay = wl.slot_layout(w1)
    flops, t_total, done = 0.0, 0.0, []
    cores = oracle.get_threads()
    masked = w.masked_rows()
    rows_per_call = 64
    n = 0
    while t_total < budget_s and n < w.layers:
        p = wl.probe_inputs(w1, n)
        t0 = time.perf_counter()
        oracle.probe_layer(p["q"], p["k_req"], p["v_req"], p["k_aff"], p["v_aff"], T=w.T, l=w.l,
                           masked_rows=masked, scale=w.scale)
        t_total += time.perf_counter() - t0
        flops += probe_flops(w1) / w.layers
        done.append(f"probe L{n}")
        if t_total >= budget_s:
            break
        r = wl.recompute_inputs(w1, n)
        rs = np.empty((1, w.T), np.int32)
        anchors = np.arange(w.K, dtype=np.int32)[None]
        _, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
        kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=w.torch_dtype)
        kc[lay.private_slots[0].long()] = r["k_new"][0]
        kc[lay.shared_slot.long()] = p["k_aff"]
        vc = torch.zeros_like(kc)
        vc[lay.private_slots[0].long()] = r["v_new"][0]
        vc[lay.shared_slot.long()] = p["v_aff"]
        rows = list(range(min(rows_per_call, w.R)))
        t0 = time.perf_counter()
        oracle.slot_attention(r["q_r"], rs, kc, vc, scale=w.scale, rows=rows)
        t_total += time.perf_counter() - t0
        flops += 4.0 * len(rows) * w.T * w.d * w.hq
        done.append(f"slot L{n} rows 0..{len(rows) - 1}")
        n += 1
    desc = (f"oracle (float64 C, OpenMP {cores} threads) on request 0: {', '.join(done[:4])}"
            f"{' ...' if len(done) > 4 else ''} ({len(done)} calls, {t_total:.1f} s)")
    return flops, t_total, cores, desc


# ----------------------------------------------------------------------------- sweep
def _per_launch_ms(fn, reps=5):
    fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def _launch_set(path):
    """Per-launch times (ms) of one layer's probe (from one call over all the path's layers,
    as a step makes it), store and slot attention for the batch."""
    ac, w, lay = path.ac, path.w, path.lay
    r0 = path.rec[0]
    probe = _per_launch_ms(lambda: ac.acache_probe_scores_layers(
        path.desc, w.batch, w.T, w.l, w.L, path.masked, w.m, *path.probe_lists(),
        [path.probe_out] * w.layers, path.scores, path.ws, path.ws_bytes)) / w.layers
    write = _per_launch_ms(lambda: ac.acache_write_slots(
        path.desc, w.batch, w.R, lay.private_slots, r0["k_new"], r0["v_new"], path.kc[0], path.vc[0],
        lay.num_slots, lay.private_begin))
    slot = _per_launch_ms(lambda: ac.acache_slot_attention(
        path.desc, w.batch, w.R, r0["q_r"], w.T, path.read_slot, path.kc[0], path.vc[0], lay.num_slots,
        path.out[0]))
    return probe, write, slot


def sweep_records(peaks, dev, full=True):
    """Per-launch measurements of the workloads other than the headline one.  Four layers are
    materialised per workload (all layers have the same shapes, so a launch's time does not
    depend on which layer it runs); whole-pass times are the per-launch times times the
    launch counts and are labelled as such.  full=False keeps the record compact: the long
    suffix's slot attention at batch 1, 4 and 32 only, and the decode figures in brief."""
    peak = peaks["bf16_tflops_sustained"]
    out = []
    for name, ratios in ((wl.DREAM_INFIX.name, (200,)), (wl.LLADA_PAGED.name, (200,)),
                         (wl.LLADA_SUFFIX.name, (100, 200, 300))):
        base = wl.CATALOGUE[name]
        for ratio in ratios:
            w = base.replace(layers=4, recompute_points=1, ratio_permille=ratio)
            path = Path(w, dev)
            path.step()
            torch.cuda.synchronize()
            probe_ms, write_ms, slot_ms = _launch_set(path)
            row = w.hkv * w.d * w.esize
            slot_tf = slot_flops_per_launch(w) / (slot_ms / 1e3) / 1e12
            probe_tf = probe_flops(w) / w.layers / (probe_ms / 1e3) / 1e12
            line = {"sweep": name, "ratio": ratio / 1000, "K": w.K, "R": w.R, "batch": w.batch, "T": w.T,
                    "layers_full": base.layers, "recompute_points_full": base.recompute_points,
                    "probe_ms_per_layer": probe_ms, "probe_tflops": probe_tf,
                    "probe_frac_of_peak": probe_tf / peak,
                    "slot_attn_ms_per_launch": slot_ms, "slot_attn_tflops": slot_tf,
                    "slot_attn_frac_of_peak": slot_tf / peak,
                    "write_ms_per_launch": write_ms,
                    "write_gbs": 4.0 * w.batch * w.R * row / (write_ms / 1e3) / 1e9,
                    "anchor_scored_tokens_per_s_est": w.batch * w.L / (base.layers * probe_ms / 1e3),
                    "full_pass_ms_est": base.layers * probe_ms + base.recompute_points * base.layers * (write_ms + slot_ms),
                    "peak": {"bf16_tflops_sustained": peak, "hbm_gbs": peaks["hbm_gbs"], "source": peaks["source"]}}
            if name in (wl.LLADA_PAGED.name, wl.DREAM_INFIX.name):
                dec = Decode(path).measure(5, 2, peaks)
                line["decode"] = dec if full else {
                    "attn_ms_per_launch": dec["attn_ms_per_launch"], "write_ms_per_launch": dec["write_ms_per_launch"],
                    "unique_gbs": dec["roofline"]["achieved"], "frac_of_hbm": dec["roofline"]["frac"]}
            if name == wl.LLADA_SUFFIX.name and ratio == 200:
                one = Path(w.replace(batch=1), dev)
                one.step()
                p1, _, _ = _launch_set(one)
                line["probe_ms_per_request_batch1"] = base.layers * p1
                del one
                vs = {}
                for b in ((1, 2, 4, 8, 16, 32) if full else (1, 4, 32)):
                    if b == w.batch:
                        vs[b] = slot_tf
                        continue
                    pb = Path(w.replace(batch=b, layers=1), dev)
                    pb.step()
                    _, _, sb = _launch_set(pb)
                    vs[b] = slot_flops_per_launch(pb.w) / (sb / 1e3) / 1e12
                    del pb
                line["slot_attn_tflops_vs_batch"] = vs
            out.append(line)
            del path
            torch.cuda.empty_cache()
    return out


def sweep(args):
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for line in sweep_records(measured_peaks(), dev):
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x, device=None):
    """Max of a per-rank float over the default process group (the timing reduction of the
    multi-GPU replicas); the identity without a process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cpu():
    """The host's CPU: os.cpu_count() and the model name lscpu reports (None if unknown)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"cpu_count": os.cpu_count(), "model": model}


def oracle_sample_step(w, layer, rows_per_layer=64, layers=4):
    """One reference-arm step: a bounded sample of the workload for the oracle -- request 0,
    `layers` consecutive layers from `layer` on, each the probe of all heads and the slot
    attention of the first `rows_per_layer` recomputed rows.  Returns (flops, seconds)."""
    import numpy as np
    import oracle
    w1 = w.replace(batch=1)
    lay = wl.slot_layout(w1)
    masked = w.masked_rows()
    flops, secs = 0.0, 0.0
    for i in range(layers):
        n = (layer + i) % w.layers
        p = wl.probe_inputs(w1, n)
        r = wl.recompute_inputs(w1, n)
        anchors = np.arange(w.K, dtype=np.int32)[None]
        _, rs = oracle.build_slot_maps(anchors, lay.shared_slot, lay.private_slots, T=w.T, l=w.l, L=w.L)
        kc = torch.zeros((lay.num_slots, w.hkv, w.d), dtype=w.torch_dtype)
        vc = torch.zeros_like(kc)
        kc[lay.private_slots[0].long()], vc[lay.private_slots[0].long()] = r["k_new"][0], r["v_new"][0]
        kc[lay.shared_slot.long()], vc[lay.shared_slot.long()] = p["k_aff"], p["v_aff"]
        rows = list(range(min(rows_per_layer, w.R)))
        t0 = time.perf_counter()
        oracle.probe_layer(p["q"], p["k_req"], p["v_req"], p["k_aff"], p["v_aff"], T=w.T, l=w.l,
                           masked_rows=masked, scale=w.scale)
        oracle.slot_attention(r["q_r"], rs, kc, vc, scale=w.scale, rows=rows)
        secs += time.perf_counter() - t0
        flops += probe_flops(w1) / w.layers + 4.0 * len(rows) * w.T * w.d * w.hq
    return flops, secs


def run_reference(args, w, world, rank):
    """The reference arm: the float64 CPU oracle, as it stands, on the host cores.  A step is a
    bounded sample of the workload (oracle_sample_step); W untimed steps, then K timed ones."""
    if rank != 0:
        return
    import oracle
    layers_per_step = 4
    for k in range(args.warmup):
        oracle_sample_step(w, k * layers_per_step, layers=layers_per_step)
    flops, secs = 0.0, 0.0
    for k in range(args.steps):
        f, t = oracle_sample_step(w, (args.warmup + k) * layers_per_step, layers=layers_per_step)
        flops += f
        secs += t
    v = flops / secs / 1e12
    cores = oracle.get_threads()
    sample = (f"one step = request 0 of the workload, {layers_per_step} layers, each the probe of all "
              f"{w.hq} heads over P = {w.P} rows and the slot attention of the first 64 of R = {w.R} "
              f"recomputed rows ({flops / args.steps / 1e9:.1f} GFLOP per step)")
    line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "step": "a bounded sample of the workload (see cpu_baseline.sample), not a full step",
            "ms_per_full_step_extrapolated": step_flops(w) / (v * 1e12) * 1e3,
            "extrapolation": "the full step's algorithmic FLOPs divided by the measured sample rate",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shapes of the LLaDA-8B prefix workload)",
            "config": {"workload": w.name, **{k: v2 for k, v2 in w.describe().items() if k != "workload"}},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample, **host_cpu()},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.sweep:
        sweep(args)
        return
    w = wl.CATALOGUE[args.workload]
    if args.layers:
        w = w.replace(layers=args.layers)
    if args.points:
        w = w.replace(recompute_points=args.points)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    path = Path(w, dev, seed_offset=rank)
    if args.decode_only:
        path.step()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps(Decode(path).measure(2, 2, measured_peaks())))
        return
    for _ in range(max(args.warmup, 3)):
        path.step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x):
        return reduce_max(x, dev)

    ev = {"select": [], "probe": []}
    clocks = ClockSampler(os.path.join(tempfile.gettempdir(), f"acache_clocks_{os.getpid()}_r{rank}.csv"))
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clocks:
        start.record()
        for _ in range(args.steps):
            path.step(ev)
        end.record()
        torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(start.elapsed_time(end))
    ms_per_step = ms / args.steps
    tflops = step_flops(w) * args.steps * world / (ms / 1e3) / 1e12
    slot_ms, slot_alone_ms = slot_launch_times(path)
    select_ms = statistics.mean(a.elapsed_time(b) for a, b in ev["select"])
    probe_ms = statistics.mean(a.elapsed_time(b) for a, b in ev["probe"])
    scored_tok_s = w.batch * w.L / (select_ms / 1e3)
    peaks = measured_peaks()
    probe_achieved = probe_flops(w) / (probe_ms / 1e3) / 1e12
    slot_achieved = slot_flops_per_launch(w) / (slot_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    traffic = profiled_traffic(["affix_kv_cache_gb300/csrc/tc_attn.cu"], w.name)

    e2e = None
    if not args.no_e2e:
        bi, bo = path.host_inputs()
        up_ms = path.upload_ms()
        n_e2e = max(1, min(args.steps, 10))
        path.upload(0)
        for k in range(4):                       # warm-up: the same pipeline
            path.step_e2e(k)
        torch.cuda.synchronize()
        barrier()
        e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # timed: step 0's upload (nothing to hide it behind), then n steps, each uploading the
        # next step's inputs while it computes (the last one has no next step)
        e_s.record()
        path.copy_stream.wait_event(e_s)
        path.upload(0)
        for k in range(n_e2e):
            path.step_e2e(k, upload_next=k + 1 < n_e2e)
        e_e.record()
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e_s.elapsed_time(e_e))
        path.use_set(0)
        # the host link is shared with the machine's other GPUs: its rate just before and just
        # after the timed steps tells whether a slow end-to-end step was the link's
        up_after = path.upload_ms()
        e2e = {"value": step_flops(w) * n_e2e * world / (ems / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": n_e2e,
               "uploaded": "every layer's probe Q and own K/V rows, and every layer's recompute-point Q and "
                           "fresh K/V (the shared affix cache is resident)",
               "read_back": "the step's importance scores, its anchors and the last layer's read-slot "
                            "attention output; the other layers' outputs stay on the device, where a "
                            "decoding engine consumes them",
               "ms_per_step": ems / n_e2e, "upload_ms_per_step": [up_ms, up_after],
               "h2d_gbs": [bi / (up_ms / 1e3) / 1e9, bi / (up_after / 1e3) / 1e9]}

    decode = None
    if not args.no_decode:
        decode = Decode(path).measure(max(args.steps, 5), 3, peaks)
    fused = store_attend_compare(path)
    copies = copy_bandwidth(path, peaks)

    others = None
    if world == 1 and not args.no_sweep:
        t0 = time.perf_counter()
        others = {"timing": "CUDA events per launch, 4 materialised layers per workload (see sweep_records)",
                  "records": sweep_records(peaks, dev, full=False)}
        others["seconds"] = time.perf_counter() - t0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops, secs, cores, desc = cpu_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc, **host_cpu()}

    if rank == 0:
        gb_touched = sum(t.numel() * t.element_size() for p in path.probe for t in p.values()) + \
            sum(t.numel() * t.element_size() for r in path.rec for t in r.values()) + \
            2 * sum(k.numel() * k.element_size() for k in path.kc)
        line = {
            "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; LLaDA-8B attention shapes, no weights or datasets)",
            "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "workload"},
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": f"inputs larger than L2: {gb_touched / 1e9:.1f} GB touched per step"},
            "anchor_scored_tokens_per_s": scored_tok_s,
            "select_ms": select_ms,
            "probe_ms": probe_ms,
            "probe_roofline": {"bound": "tensor", "kernel": "probe (forward + mass + head sum, all layers, "
                                                           "one chained call)",
                               "achieved": probe_achieved, "peak": peaks["bf16_tflops_sustained"],
                               "unit": "TFLOP/s", "frac": probe_achieved / peaks["bf16_tflops_sustained"],
                               "flops": "the forward's 4·P·T·d per row-head-layer only (the mass pass's "
                                        "2·m·L·d recompute not counted)",
                               "peak_source": f"{peaks['source']} bf16 sustained"},
            "slot_attn_ms_per_launch": slot_ms,
            "slot_attn_timing": "per launch within one call over all layers (launches chained); "
                                "slot_attn_ms_per_launch_alone: one launch at a time",
            "slot_attn_ms_per_launch_alone": slot_alone_ms,
            "roofline": {"bound": "tensor", "kernel": "slot_attention", "achieved": slot_achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": slot_achieved / peak,
                         "peak_source": f"{peaks['source']} bf16 sustained", "traffic": traffic},
            "decode": decode,
            "store_then_attend": {"timing": "CUDA events, one recompute point over all layers, 3 passes",
                                  **fused},
            "copies": {"timing": "CUDA events, every layer, 3 passes", **copies},
            "other_workloads": others,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": path.launches_per_step * args.steps,
            "clocks": clocks.summary(local),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
