"""Benchmark of the block-quantized decode path on GB300.

Default workload (the headline): the full dense 8B-class decode step with
Q4_K weights -- 32 layers (q 4096x4096, k/v 1024x4096, o 4096x4096, gate/up
2x14336x4096 with SwiGLU, down 4096x14336, weightless RMS pre-norms, a
one-token-context attention stand-in) plus the 128256x4096 LM head, batch 1
(--nvec 2/4/8 for speculative-verify columns).  One "step" = one token
through all 129 dequant-GEMVs, replayed from one CUDA graph.  4.2 GB of
packed weights stay resident and every step streams all of them, far beyond
the 129 MB L2, so no flush is needed.

Other workloads (--workload): gemv4096 (the single Q4_K 4096x4096
dequant-GEMV, rotated over ceil(4 L2 / 9.4 MB) = 55 copies per step so that no
launch finds its weights in L2); moe_decode (40 MoE layers, hidden 2048, 256
experts of gate/up 512x2048 + down 2048x512, top-8 + shared expert, Zipf(1.1)
routing, a 64-token decode run per step); moe_layer (one MoE layer of hidden
4096 with 512 experts of gate/up 2x1024x4096 + down 4096x1024, top-4 + shared
expert, --ntok 1 or 8 tokens per forward; value = effective weight GB/s).
The default run also measures gemv4096, moe_layer (1 and 8 tokens) and
moe_decode and reports each as a sub-object of the headline line
(--no-sub skips them).  --chain runs the dense step as one epq_gemv_chain
launch instead of one launch per matrix.

The JSON line carries: value (tok/s for decode workloads, GB/s otherwise),
the mean over the K bracketed steps plus the median and minimum of K
individually timed replays, the roofline of the dominant kernel (its time
per launch from a graph of back-to-back launches of that kernel alone on
distinct weights, programmatic dependent launch as in the step), e2e (host
buffers, H2D + D2H inside the timed region), clocks sampled every 100 ms
while the step replays back to back before, during and after the timed
region, gpu_launches, and the CPU baseline: the plain C++ oracle's float32
dequant-GEMV at 1 thread and at all host threads (guided row split) on a
bounded sample.  --impl reference times that oracle itself, one bounded
sample per step.
"""
from __future__ import annotations

import argparse
import datetime
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective weight GB/s and % of HBM peak for Q4_K dequant-GEMV; decode tok/s"
NOMINAL_HBM_GBS = 8000.0
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the kernel as it stands; the summary with its command is the
# named file.  An entry must go when its kernel changes.
NCU_TRAFFIC = {
    ("moe_decode", "moe_gateup"): (10_683_904, "profiles/moe_tc_gateup_down_q4k_full.md"),
    ("dense8b", "gemv_gateup"): (66_589_696, "profiles/gemv_k16_q4k_dense8b_full.md"),
}
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms.  The
    summary keeps the samples stamped inside the window between mark_start()
    and mark_end() (all of them if the stamps cannot be read)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")
    INTERVAL_MS = 100

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t_start = None
        self.t_end = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    @staticmethod
    def _stamp(text):
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                continue
        return None

    def parse(self, lines):
        """(sm MHz, max MHz, reasons, stamp or None) for each sample line."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        out = []
        for line in lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, smax = float(f[1]), float(f[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, f[5:9]) if v.lower() == "active"}
            out.append((sm, smax, reasons, self._stamp(f[9]) if len(f) > 9 else None))
        return out

    def summary(self):
        try:
            rows = self.parse(open(self.path))
        except Exception:
            rows = []
        window = None
        if self.t_start is not None and self.t_end is not None and rows and all(r[3] is not None for r in rows):
            inside = [r for r in rows if self.t_start <= r[3] <= self.t_end]
            if inside:
                rows, window = inside, round(self.t_end - self.t_start, 3)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        out = {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
               "reasons": sorted(set().union(*(r[2] for r in rows))), "samples": len(rows)}
        if window is not None:
            out["window_s"] = window
            out["sampled"] = (f"every {self.INTERVAL_MS} ms while the GPU replayed the step back to back "
                              "before, during and after the timed region")
        return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v, device="cpu"):
    """The largest v over the ranks of the process group (a job's time is its
    slowest rank's); v itself without a group or with a single rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, n_ranks, ms):
    """Whole-job throughput: the units every rank processed over the slowest rank's time (ms)."""
    return units_per_rank * n_ranks / (ms * 1e-3)


# ------------------------------------------------------------------ workloads
class Workload:
    name = ""
    unit = "tok/s"
    units_per_step = 1.0       # tokens (or bytes) per step
    dtype = "f32"

    def config(self):
        return {}


def quantize_into(epq, fmt, W, out=None):
    return epq.epq_quantize(fmt, W, blocks=out)


FMT_TAG = {0: "q8_0", 1: "q4_0", 2: "q4_1", 3: "q4k", 4: "q2k", 5: "q6k"}


class Gemv4096Workload(Workload):
    """The single dequant-GEMV (Q4_K unless another format is named) (W 4096x4096 Student-t(5)*0.02, x ~ N(0,1),
    batch 1), one launch per copy over ceil(4 L2 / row bytes) copies of the
    packed matrix, so every launch streams its 9.4 MB from HBM.  Launches are
    chained with programmatic dependent launch as in a decode step (the
    weights stream while the previous launch drains)."""
    name = "gemv4096"
    unit = "GB/s"

    def __init__(self, epq, dev, fmt, nvec=1):
        import torch
        from synthetic import workloads as wl
        self.fmt, self.dev, self.epq, self.nvec = fmt, dev, epq, nvec
        n = 4096
        packed = epq.epq_quantize(fmt, wl.weight("gemv4096", 0, 0, n, n, dev))
        self.matrix_bytes = packed.numel()
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.copies = max(2, math.ceil(4 * l2 / self.matrix_bytes))
        self.W = packed.unsqueeze(0).repeat(self.copies, 1, 1).contiguous()
        self.x = wl.activations("gemv4096", nvec, n, dev)
        self.out = torch.empty((self.copies, nvec, n), dtype=torch.float32, device=dev)
        self.bytes_per_launch = self.matrix_bytes + 4 * nvec * (n + n)
        self.units_per_step = self.copies * self.matrix_bytes / 1e9         # weight GB per step
        self.kernels_per_step = self.copies
        self.kernel_bytes = {"gemv4096": self.bytes_per_launch}
        self.launches = {"gemv4096": self.copies}
        self.full_step_bytes = self.copies * self.matrix_bytes

    def config(self):
        return {"workload": f"gemv4096_{FMT_TAG[self.fmt]}", "rows": 4096, "cols": 4096, "nvec": self.nvec, "batch": 1,
                "packed_bytes": self.matrix_bytes, "copies_per_step": self.copies,
                "l2": f"{self.copies} rotating copies ({self.copies * self.matrix_bytes / 1e6:.0f} MB > 4x L2)"}

    def step(self, stream, x=None, out=None, timers=None):
        x = self.x if x is None else x
        out = self.out if out is None else out
        for c in range(self.copies):
            self.epq.epq_gemv_ex(self.fmt, self.W[c], x, 4096, 4096, y=out[c], weights_ready=True, stream=stream)

    def kernel_bench(self, name):
        return (lambda s: self.step(s)), self.copies

    def cpu_mats(self):
        return [(self.W[0].cpu().numpy(), 4096)], self.full_step_bytes


class MoEDecodeWorkload(Workload):
    name = "moe_decode"
    unit = "tok/s"

    def __init__(self, epq, dev, fmt, layers=None, attn_ctx=None, expert_fmt=None, down_fmt=None):
        from synthetic import workloads as wl
        self.cfg = c = wl.MoEDecode() if layers is None else wl.MoEDecode(layers=layers)
        self.attn_ctx = attn_ctx
        self.fmt, self.dev, self.epq = fmt, dev, epq
        # expert formats: gate/up (and down unless down_fmt is given); attention projections stay in fmt
        self.efmt = fmt if expert_fmt is None else expert_fmt
        self.dfmt = self.efmt if down_fmt is None else down_fmt
        H, I, E = c.hidden, c.inter, c.n_experts
        rbH, rbI = epq.epq_row_bytes(fmt, H), epq.epq_row_bytes(fmt, I)
        erbH, drbI = epq.epq_row_bytes(self.efmt, H), epq.epq_row_bytes(self.dfmt, I)
        import torch
        self.layers = []
        for l in range(c.layers):
            wqkv = torch.empty((3 * H, rbH), dtype=torch.uint8, device=dev)
            for t in range(3):
                epq.epq_quantize(fmt, wl.weight("moe_decode", l, t, H, H, dev), blocks=wqkv[t * H:(t + 1) * H])
            wo = epq.epq_quantize(fmt, wl.weight("moe_decode", l, 3, H, H, dev))
            R, bias = wl.moe_router("moe_decode", l, E, H, dev, c.zipf_s)
            gu = torch.empty((E, 2 * I, erbH), dtype=torch.uint8, device=dev)
            dn = torch.empty((E, H, drbI), dtype=torch.uint8, device=dev)
            for e0 in range(0, E, 64):
                n = min(64, E - e0)
                Wg = wl.weight("moe_decode", l, 10, n * 2 * I, H, dev, expert=e0)
                epq.epq_quantize(self.efmt, Wg, blocks=gu[e0:e0 + n].view(n * 2 * I, erbH))
                Wd = wl.weight("moe_decode", l, 11, n * H, I, dev, expert=e0)
                epq.epq_quantize(self.dfmt, Wd, blocks=dn[e0:e0 + n].view(n * H, drbI))
                del Wg, Wd
            sgu = epq.epq_quantize(self.efmt, wl.weight("moe_decode", l, 12, 2 * I, H, dev))
            sdn = epq.epq_quantize(self.dfmt, wl.weight("moe_decode", l, 13, H, I, dev))
            layer = epq.MoELayer(self.efmt, R, gu, dn, router_bias=bias, shared_gate_up=sgu, shared_down=sdn,
                                 down_fmt=self.dfmt)
            self.layers.append((wqkv, wo, layer))
        torch.cuda.synchronize()
        from moe_experts_gb300.decode import MoEDecoder
        self.model = MoEDecoder(c, fmt, self.layers, dev, attn_ctx=attn_ctx, max_new=c.tokens)
        self.T = c.tokens
        self.x = wl.activations("moe_decode", self.T, H, dev)
        self.out = torch.empty((self.T, H), dtype=torch.float32, device=dev)
        self.units_per_step = float(self.T)
        self.bytes_per_token = c.layers * (4 * H * rbH + E * H * 4 + (c.topk + 1) * (2 * I * erbH + H * drbI))
        self.kernels_per_step = self.T * c.layers * (5 if attn_ctx is None else 6)
        self.launches = {k: self.T * c.layers for k in ("gemv_qkv", "gemv_o", "moe_router", "moe_gateup",
                                                          "moe_down")}
        if attn_ctx is not None:
            self.launches["attention"] = self.T * c.layers
        # dominant-kernel candidates: name -> algorithmic bytes per launch
        self.kernel_bytes = {
            "gemv_qkv": 3 * H * rbH + 4 * (H + 3 * H),
            "gemv_o": H * rbH + 4 * (H + 2 * H),
            "moe_router": E * H * 4 + 4 * H,
            "moe_gateup": (c.topk + 1) * 2 * I * erbH + 4 * (H + (c.topk + 1) * I),
            "moe_down": (c.topk + 1) * H * drbI + 4 * ((c.topk + 1) * I + 2 * H),
        }
        if attn_ctx is not None:  # an upper bound: value rows of skipped positions are not read
            self.kernel_bytes["attention"] = 2 * c.heads * (attn_ctx + c.tokens // 2) * epq.epq_kv_row_bytes(
                c.head_dim) + 4 * 4 * H

    def config(self):
        c = self.cfg
        tag = FMT_TAG[self.efmt] + ("" if self.dfmt == self.efmt else f"_{FMT_TAG[self.dfmt]}down")
        return {"workload": f"moe_decode_{tag}" + ("" if self.attn_ctx is None else f"_attn{self.attn_ctx}"),
                "expert_formats": {"gate_up": FMT_TAG[self.efmt], "down": FMT_TAG[self.dfmt],
                                   "attention_projections": FMT_TAG[self.fmt]},
                "attention": "one-token-context stand-in" if self.attn_ctx is None else
                f"Q8_0 KV cache, {self.attn_ctx} cached positions + the 64-token run, ln(1e-4) skip threshold",
                "layers": c.layers, "hidden": c.hidden, "experts": c.n_experts,
                "inter": c.inter, "topk": c.topk, "shared_experts": 1, "tokens_per_step": c.tokens, "batch": 1,
                "router": "fp32 zipf(1.1)", "weights_resident_gb": round(self.resident_gb(), 2),
                "bytes_per_token": self.bytes_per_token,
                "l2": f"inputs larger than L2 ({self.bytes_per_token / 1e9:.2f} GB/token)"}

    def resident_gb(self):
        tot = 0
        for wqkv, wo, layer in self.layers:
            tot += wqkv.numel() + wo.numel() + layer.gate_up.numel() + layer.down.numel()
            tot += layer.router.numel() * 4 + layer.shared_gate_up.numel() + layer.shared_down.numel()
        return tot / 1e9

    def step(self, stream, x=None, out=None, timers=None):
        x = self.x if x is None else x
        out = self.out if out is None else out
        for t in range(self.T):
            self.model.token(x[t:t + 1], out[t:t + 1], stream=stream, timers=timers if t < 64 else None,
                             pos=None if self.attn_ctx is None else self.attn_ctx + t)

    def kernel_bench(self, name):
        """One launch of the named kernel per layer (40 back to back, each
        layer's own weights) on the decoder's buffers."""
        e, c, f, H = self.epq, self.cfg, self.fmt, self.cfg.hidden
        m = self.model
        st = {"moe_router": e.EPQ_MOE_ROUTE, "moe_gateup": e.EPQ_MOE_GATE_UP, "moe_down": e.EPQ_MOE_DOWN}

        def run(s):
            for li, (wqkv, wo, moe) in enumerate(self.layers):
                if name == "attention":
                    q = m.qkv[0]
                    e.epq_attention_decode(q[:H], q[H:2 * H], q[2 * H:], m.caches[li], c.heads, self.attn_ctx,
                                           1.0 / math.sqrt(c.head_dim), math.log(1e-4), out=m.attn[0], stream=s)
                elif name == "gemv_qkv":
                    e.epq_gemv_ex(f, wqkv, m.h, 3 * H, H, y=m.qkv, rms_prenorm=True, rms_eps=c.rms_eps,
                                  weights_ready=True, stream=s)
                elif name == "gemv_o":
                    e.epq_gemv_ex(f, wo, m.qkv[:, 2 * H:] if self.attn_ctx is None else m.attn, H, H,
                                  y=self.out[:1], residual=m.h, weights_ready=True, stream=s)
                else:
                    e.epq_moe_forward(moe, m.h, c.topk, y=self.out[:1], workspace=m.ws, rms_prenorm=True,
                                      rms_eps=c.rms_eps, stages=st[name], stream=s)
        return run, c.layers

    def routing_report(self, stream):
        """Realised expert popularity of one 64-token run (untimed): per layer,
        the experts' selection counts ranked, pooled over layers; the slope of
        log(count) on log(rank) over the experts chosen at least once."""
        import numpy as np
        import torch
        c = self.cfg
        idx = torch.empty((self.T, c.layers, c.topk), dtype=torch.int32, device=self.dev)
        with torch.cuda.stream(stream):
            for t in range(self.T):
                self.model.token(self.x[t:t + 1], self.out[t:t + 1], stream=stream, idx_out=idx[t],
                                 pos=None if self.attn_ctx is None else self.attn_ctx + t)
        stream.synchronize()
        sel = idx.cpu().numpy()
        ranked = np.zeros(c.n_experts)
        touched = []
        for l in range(c.layers):
            cnt = np.bincount(sel[:, l, :].reshape(-1), minlength=c.n_experts)
            touched.append(int((cnt > 0).sum()))
            ranked += np.sort(cnt)[::-1]
        ranked /= c.layers
        r = np.arange(1, c.n_experts + 1)
        keep = ranked > 0
        slope = float(np.polyfit(np.log(r[keep]), np.log(ranked[keep]), 1)[0])
        return {"selections_per_layer": self.T * c.topk, "experts_touched_per_layer_avg": round(float(np.mean(touched)), 1),
                "rank_frequency_top10": [round(float(v), 2) for v in ranked[:10]],
                "rank_frequency_at_rank_50_100_150": [round(float(ranked[i]), 2) for i in (49, 99, 149)],
                "fitted_log_log_slope": round(slope, 3), "router_zipf_s": c.zipf_s}

    # ---- oracle on a bounded sample (a few layers of one token)
    def oracle_sample(self, budget_s=20.0):
        import numpy as np
        import oracle
        from oracle.moe import MoEWeights
        c = self.cfg
        H, I = c.hidden, c.inter
        x = self.x[0:1].cpu().numpy().astype(np.float32)
        h = x.astype(np.float64)
        t0 = time.perf_counter()
        done = 0
        for l, (wqkv, wo, layer) in enumerate(self.layers):
            pq = wqkv.cpu().numpy()
            po = wo.cpu().numpy()
            mw = MoEWeights(fmt=self.fmt, hidden=H, inter=I, router=layer.router.cpu().numpy(),
                            gate_up=None, down=None, router_bias=layer.router_bias.cpu().numpy(),
                            shared_gate_up=layer.shared_gate_up.cpu().numpy(),
                            shared_down=layer.shared_down.cpu().numpy())
            ts = time.perf_counter()
            xn = oracle.rmsnorm_f64(h, c.rms_eps)
            qkv = oracle.gemv_f64(self.fmt, pq, xn, H)
            h = h + oracle.gemv_f64(self.fmt, po, qkv[:, 2 * H:], H)
            xin = oracle.rmsnorm_f64(h, c.rms_eps)
            logits = oracle.router_logits_f64(mw.router, xin, mw.router_bias)
            idx = oracle.topk_select(logits, c.topk)
            w = oracle.combine_weights(logits, idx, True)
            y = h.copy()
            gu_all, dn_all = layer.gate_up, layer.down
            for k, e in enumerate(idx[0]):
                o = oracle.expert_forward_f64(self.efmt, gu_all[int(e)].cpu().numpy(), dn_all[int(e)].cpu().numpy(),
                                              H, I, xin[0], self.dfmt)[0]
                y += w[0, k] * o
            o = oracle.expert_forward_f64(self.efmt, mw.shared_gate_up, mw.shared_down, H, I, xin[0], self.dfmt)[0]
            h = y + o
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        per_token = dt / done * c.layers
        return 1.0 / per_token, f"1 token through {done} of {c.layers} layers (oracle, float64), scaled to 40 layers"


class MoELayerWorkload(Workload):
    """One MoE layer (hidden 4096, 512 experts of gate/up 2x1024x4096 + down
    4096x1024, Q4_K, 3.6 GB resident; one shared expert; router 512x4096
    fp32; top-4), ntok tokens per forward.  A step is one forward on each of
    `replicas` (router, shared expert, x) sets that share the routed experts:
    the replicas' routers and shared experts together exceed 4x L2, and each
    x routes differently, so no forward finds its weights in L2 except by
    chance (a routed expert chosen again within the last ~3 forwards)."""
    name = "moe_layer"
    unit = "GB/s"

    def __init__(self, epq, dev, fmt, ntok=1, replicas=None):
        import torch
        from synthetic import workloads as wl
        self.cfg = c = wl.MoELayer()
        self.fmt, self.dev, self.epq, self.ntok = fmt, dev, epq, ntok
        H, I, E, K = c.hidden, c.inter, c.n_experts, c.topk
        rbH, rbI = epq.epq_row_bytes(fmt, H), epq.epq_row_bytes(fmt, I)
        self.expert_bytes = 2 * I * rbH + H * rbI
        gu = torch.empty((E, 2 * I, rbH), dtype=torch.uint8, device=dev)
        dn = torch.empty((E, H, rbI), dtype=torch.uint8, device=dev)
        for e in range(E):  # one generator call per expert (the tests regenerate single experts)
            epq.epq_quantize(fmt, wl.weight("moe_layer", 0, 10, 2 * I, H, dev, expert=e), blocks=gu[e])
            epq.epq_quantize(fmt, wl.weight("moe_layer", 0, 11, H, I, dev, expert=e), blocks=dn[e])
        per_rep = E * H * 4 + self.expert_bytes
        self.R = replicas if replicas else max(1, math.ceil(4 * 129e6 / per_rep))
        self.layers = []
        for r in range(self.R):
            Rw, _ = wl.moe_router("moe_layer", r, E, H, dev, None)
            sgu = epq.epq_quantize(fmt, wl.weight("moe_layer", r, 12, 2 * I, H, dev))
            sdn = epq.epq_quantize(fmt, wl.weight("moe_layer", r, 13, H, I, dev))
            self.layers.append(epq.MoELayer(fmt, Rw, gu, dn, shared_gate_up=sgu, shared_down=sdn))
        self.gate_up, self.down = gu, dn
        self.x = torch.stack([wl.activations("moe_layer", ntok, H, dev, stream_id=r) for r in range(self.R)])
        self.out = torch.empty_like(self.x)
        self.ws = torch.empty(self.layers[0].workspace_bytes(ntok, K), dtype=torch.uint8, device=dev)
        # distinct routed experts of each forward (the bytes it must stream)
        idx = torch.empty((ntok, K), dtype=torch.int32, device=dev)
        self.distinct = []
        # Q4_K calls of more than two tokens run as chunks of two (router,
        # gate/up, down per chunk): the launches, and the bytes each streams
        self.chunks = [(0, ntok)] if (ntok <= 2 or fmt != epq.EPQ_Q4_K) else \
            [(t0, min(2, ntok - t0)) for t0 in range(0, ntok, 2)]
        chunk_distinct = []
        for r in range(self.R):
            epq.epq_moe_forward(self.layers[r], self.x[r], K, y=self.out[r], topk_idx=idx, workspace=self.ws)
            ids = idx.cpu().tolist()
            self.distinct.append(len({e for row in ids for e in row}))
            for t0, nt in self.chunks:
                chunk_distinct.append(len({e for row in ids[t0:t0 + nt] for e in row}))
        torch.cuda.synchronize()
        nd = sum(self.distinct) / self.R
        ndc = sum(chunk_distinct) / len(chunk_distinct)
        ntc = ntok / len(self.chunks)
        act = 4 * ntok * H * 2  # x in, y out
        self.bytes_per_forward = E * H * 4 + (nd + 1) * self.expert_bytes + act
        self.units_per_step = self.R * self.bytes_per_forward / 1e9   # GB per step
        self.tokens_per_step = self.R * ntok
        self.kernels_per_step = 3 * self.R * len(self.chunks)
        self.launches = {k: self.R * len(self.chunks) for k in ("moe_router", "moe_gateup", "moe_down")}
        # algorithmic bytes of one launch of each kernel (per chunk)
        self.kernel_bytes = {
            "moe_router": E * H * 4 + 4 * ntc * H,
            "moe_gateup": (ndc + 1) * 2 * I * rbH + 4 * ntc * (H + (K + 1) * I),
            "moe_down": (ndc + 1) * H * rbI + 4 * ntc * ((K + 1) * I + 2 * H),
        }

    def config(self):
        c = self.cfg
        return {"workload": "moe_layer_q4k", "hidden": c.hidden, "experts": c.n_experts, "inter": c.inter,
                "topk": c.topk, "shared_experts": 1, "ntok": self.ntok, "forwards_per_step": self.R,
                "token_chunks_per_forward": len(self.chunks),
                "distinct_routed_experts_avg": round(sum(self.distinct) / self.R, 2),
                "bytes_per_forward": int(self.bytes_per_forward), "router": "fp32 student-t",
                "l2": f"{self.R} router+shared replicas ({self.R * (c.n_experts * c.hidden * 4 + self.expert_bytes) / 1e6:.0f}"
                      " MB > 4x L2), x per replica, routed experts drawn from 3.6 GB"}

    def step(self, stream, x=None, out=None, timers=None):
        x = self.x if x is None else x
        out = self.out if out is None else out
        e, K = self.epq, self.cfg.topk
        for r in range(self.R):
            if timers is None:
                e.epq_moe_forward(self.layers[r], x[r], K, y=out[r], workspace=self.ws, stream=stream)
                continue
            # the same kernels per chunk as the plain call, one stage per call
            for t0, nt in self.chunks:
                for name, st in (("moe_router", e.EPQ_MOE_ROUTE), ("moe_gateup", e.EPQ_MOE_GATE_UP),
                                 ("moe_down", e.EPQ_MOE_DOWN)):
                    a, b = timers.pair(name)
                    a.record(stream)
                    e.epq_moe_forward(self.layers[r], x[r][t0:t0 + nt], K, y=out[r][t0:t0 + nt], workspace=self.ws,
                                      stages=st, stream=stream)
                    b.record(stream)

    def kernel_bench(self, name):
        """The named stage of every chunk of every replica's forward, back to
        back (the same kernels as the timed call)."""
        e, K = self.epq, self.cfg.topk
        st = {"moe_router": e.EPQ_MOE_ROUTE, "moe_gateup": e.EPQ_MOE_GATE_UP, "moe_down": e.EPQ_MOE_DOWN}[name]

        def run(s):
            for r in range(self.R):
                for t0, nt in self.chunks:
                    e.epq_moe_forward(self.layers[r], self.x[r][t0:t0 + nt], K, y=self.out[r][t0:t0 + nt],
                                      workspace=self.ws, stages=st, stream=s)
        return run, self.R * len(self.chunks)

    def extra(self, value):
        return {"tok_per_s": round(value / self.bytes_per_forward * 1e9 * self.ntok, 1),
                "us_per_forward": round(self.bytes_per_forward / (value * 1e9) * 1e6, 3)}

    def oracle_sample(self, budget_s=20.0):
        import numpy as np
        import oracle
        c = self.cfg
        H, I, K = c.hidden, c.inter, c.topk
        layer = self.layers[0]
        R = layer.router.cpu().numpy()
        sgu, sdn = layer.shared_gate_up.cpu().numpy(), layer.shared_down.cpu().numpy()
        xs = self.x[0].cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        nbytes, done = 0, 0
        while True:
            x = xs[done % self.ntok]
            logits = oracle.router_logits_f64(R, x[None], None)
            idx = oracle.topk_select(logits, K)
            w = oracle.combine_weights(logits, idx, True)
            y = x.copy()
            for k, ex in enumerate(idx[0]):
                o = oracle.expert_forward_f64(self.fmt, self.gate_up[int(ex)].cpu().numpy(),
                                              self.down[int(ex)].cpu().numpy(), H, I, x)[0]
                y += w[0, k] * o[0]
            y += oracle.expert_forward_f64(self.fmt, sgu, sdn, H, I, x)[0][0]
            nbytes += R.nbytes + (K + 1) * self.expert_bytes
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return nbytes / dt / 1e9, f"{done} single-token forwards of the layer (oracle, float64), router + {K} + 1 experts each"


class DenseDecodeWorkload(Workload):
    name = "dense8b"
    unit = "tok/s"

    def __init__(self, epq, dev, fmt, nvec=1, layers=None, chain=False, attn_ctx=None):
        import torch
        from synthetic import workloads as wl
        self.cfg = c = wl.DenseDecode() if layers is None else wl.DenseDecode(layers=layers)
        self.attn_ctx = attn_ctx if (nvec == 1 and not chain) else None
        self.fmt, self.dev, self.epq, self.nvec = fmt, dev, epq, nvec
        H = c.hidden
        rbH, rbI = epq.epq_row_bytes(fmt, H), epq.epq_row_bytes(fmt, c.inter)
        nq, nkv = c.q_rows, c.kv_rows
        self.layers = []
        for l in range(c.layers):
            wqkv = torch.empty((nq + 2 * nkv, rbH), dtype=torch.uint8, device=dev)
            epq.epq_quantize(fmt, wl.weight("dense8b", l, 0, nq, H, dev), blocks=wqkv[:nq])
            epq.epq_quantize(fmt, wl.weight("dense8b", l, 1, nkv, H, dev), blocks=wqkv[nq:nq + nkv])
            epq.epq_quantize(fmt, wl.weight("dense8b", l, 2, nkv, H, dev), blocks=wqkv[nq + nkv:])
            wo = epq.epq_quantize(fmt, wl.weight("dense8b", l, 3, H, nq, dev))
            wgu = torch.empty((2 * c.inter, rbH), dtype=torch.uint8, device=dev)
            epq.epq_quantize(fmt, wl.weight("dense8b", l, 4, c.inter, H, dev), blocks=wgu[:c.inter])
            epq.epq_quantize(fmt, wl.weight("dense8b", l, 5, c.inter, H, dev), blocks=wgu[c.inter:])
            wd = epq.epq_quantize(fmt, wl.weight("dense8b", l, 6, H, c.inter, dev))
            self.layers.append((wqkv, wo, wgu, wd))
        head = torch.empty((c.vocab, rbH), dtype=torch.uint8, device=dev)
        for r0 in range(0, c.vocab, 16384):
            n = min(16384, c.vocab - r0)
            epq.epq_quantize(fmt, wl.weight("dense8b", 0, 7, n, H, dev, expert=r0), blocks=head[r0:r0 + n])
        self.head = head
        torch.cuda.synchronize()
        from moe_experts_gb300.decode import DenseDecoder
        self.model = DenseDecoder(c, fmt, self.layers, head, dev, nvec=nvec, chain=chain, attn_ctx=self.attn_ctx)
        self.scratch = torch.empty((nvec, H), dtype=torch.float32, device=dev)
        self.chain = chain
        self.x = wl.activations("dense8b", nvec, H, dev)
        self.units_per_step = float(nvec)
        wbytes = c.layers * ((nq + 2 * nkv) * rbH + H * epq.epq_row_bytes(fmt, nq) + 2 * c.inter * rbH
                             + H * rbI) + c.vocab * rbH
        self.weight_bytes_per_step = wbytes
        self.bytes_per_token = wbytes / nvec  # one weight pass serves all nvec columns
        # packed bytes of the full step (the oracle's rate is scaled to it even
        # when fewer layers are built, as in the reference arm)
        full = wl.DenseDecode()
        self.full_step_bytes = full.layers * ((nq + 2 * nkv) * rbH + H * epq.epq_row_bytes(fmt, nq) +
                                              2 * c.inter * rbH + H * rbI) + c.vocab * rbH
        self.kernels_per_step = 1 if chain else c.layers * (4 if self.attn_ctx is None else 5) + 1
        self.launches = {"gemv_chain": 1} if chain else {"gemv_qkv": c.layers, "gemv_o": c.layers,
                                                          "gemv_gateup": c.layers, "gemv_down": c.layers,
                                                          "gemv_head": 1}
        if chain:  # the one launch is the dominant (and only) kernel
            self.kernel_bytes = {"gemv_chain": wbytes + 4 * nvec * (c.layers * (4 * H + 2 * c.inter + nq + 2 * nkv
                                                                                 + H) + H + c.vocab)}
        else:
            self.kernel_bytes = {
                "gemv_qkv": (nq + 2 * nkv) * rbH + 4 * nvec * (H + nq + 2 * nkv),
                "gemv_o": H * epq.epq_row_bytes(fmt, nq) + 4 * nvec * (nkv + 2 * H),
                "gemv_gateup": 2 * c.inter * rbH + 4 * nvec * (H + c.inter),
                "gemv_down": H * rbI + 4 * nvec * (c.inter + 2 * H),
                "gemv_head": c.vocab * rbH + 4 * nvec * (H + c.vocab),
            }
            if self.attn_ctx is not None:
                # key and value rows of every cached position and the step's own (value rows of skipped
                # positions are not read, so this is an upper bound of the bytes streamed)
                self.kernel_bytes["attention"] = 2 * c.kv_heads * (self.attn_ctx + 1) * epq.epq_kv_row_bytes(
                    c.head_dim) + 4 * (2 * nq + 2 * nkv)
                self.launches["attention"] = c.layers

    def config(self):
        c = self.cfg
        return {"workload": f"dense8b_decode_{'q4k' if self.fmt == 3 else self.fmt}" +
                ("" if self.attn_ctx is None else f"_attn{self.attn_ctx}"),
                "attention": "one-token-context stand-in" if self.attn_ctx is None else
                f"Q8_0 KV cache, {self.attn_ctx} cached positions, ln(1e-4) skip threshold", "layers": c.layers,
                "launch": "one epq_gemv_chain launch per step" if self.chain else "one launch per matrix",
                "hidden": c.hidden, "inter": c.inter, "heads": c.heads, "kv_heads": c.kv_heads, "vocab": c.vocab,
                "nvec": self.nvec, "batch": 1, "weight_bytes_per_step": self.weight_bytes_per_step,
                "l2": "inputs larger than L2 (4.2 GB/step)"}

    def step(self, stream, x=None, out=None, timers=None):
        self.model.step(self.x if x is None else x, stream=stream, timers=timers)

    def kernel_bench(self, name):
        """The named projection of every layer back to back (each layer's own
        weights, programmatic dependent launch as in the step) on the
        decoder's buffers; the LM head four times."""
        e, c, f, H = self.epq, self.cfg, self.fmt, self.cfg.hidden
        m = self.model
        nq, nkv = c.q_rows, c.kv_rows
        if name == "gemv_chain":
            return (lambda s: self.step(s)), 1

        def run(s):
            if name == "attention":
                q = m.qkv[0]
                for li in range(c.layers):
                    e.epq_attention_decode(q[:nq], q[nq:nq + nkv], q[nq + nkv:], m.caches[li], c.heads, m.pos,
                                           1.0 / math.sqrt(c.head_dim), math.log(1e-4), out=m.attn[0], stream=s)
                return
            if name == "gemv_head":
                for _ in range(4):
                    e.epq_gemv_ex(f, self.head, m.h, c.vocab, H, y=m.logits, rms_prenorm=True, rms_eps=c.rms_eps,
                                  weights_ready=True, stream=s)
                return
            for wqkv, wo, wgu, wd in self.layers:
                if name == "gemv_qkv":
                    e.epq_gemv_ex(f, wqkv, m.h, nq + 2 * nkv, H, y=m.qkv, rms_prenorm=True, rms_eps=c.rms_eps,
                                  weights_ready=True, stream=s)
                elif name == "gemv_o" and self.attn_ctx is not None:
                    e.epq_gemv_ex(f, wo, m.attn, H, nq, y=self.scratch, residual=m.h, weights_ready=True, stream=s)
                elif name == "gemv_o":
                    e.epq_gemv_ex(f, wo, m.qkv[:, nq + nkv:], H, nq, y=self.scratch, residual=m.h,
                                  x_group=c.heads // c.kv_heads, x_head_dim=c.head_dim, weights_ready=True, stream=s)
                elif name == "gemv_gateup":
                    e.epq_gemv_ex(f, wgu, m.h, 2 * c.inter, H, y=m.m, rms_prenorm=True, rms_eps=c.rms_eps,
                                  swiglu=True, weights_ready=True, stream=s)
                elif name == "gemv_down":
                    e.epq_gemv_ex(f, wd, m.m, H, c.inter, y=self.scratch, residual=m.h, weights_ready=True, stream=s)
        return run, (4 if name == "gemv_head" else c.layers)

    def cpu_mats(self):
        """A bounded sample for the CPU oracle: layer 0's four projections and
        1/16 of the LM head rows (packed bytes and columns each)."""
        c = self.cfg
        wqkv, wo, wgu, wd = self.layers[0]
        mats = [(wqkv.cpu().numpy(), c.hidden), (wo.cpu().numpy(), c.q_rows), (wgu.cpu().numpy(), c.hidden),
                (wd.cpu().numpy(), c.inter), (self.head[:c.vocab // 16].cpu().numpy(), c.hidden)]
        return mats, self.full_step_bytes


# ------------------------------------------------------------------ CPU oracle
def cpu_gemv_rate(fmt, mats, budget_s, threads):
    """Bytes/s of the C++ oracle's float32 dequant-GEMV over the sample
    matrices (packed uint8 [rows, row_bytes], cols), repeated until the
    budget is spent; returns (bytes per second, passes over the sample)."""
    import numpy as np
    from oracle import cref
    xs = [np.random.default_rng(7).standard_normal((1, cols)).astype(np.float32) for _, cols in mats]
    ys = [np.empty((1, p.shape[0]), np.float32) for p, _ in mats]
    nbytes, passes = 0, 0
    t0 = time.perf_counter()
    while True:
        for (p, cols), x, y in zip(mats, xs, ys):
            cref.gemv_f32(fmt, p, x, cols, threads=threads, out=y)
            nbytes += p.size
        passes += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return nbytes / (time.perf_counter() - t0), passes


def cpu_baseline_gemv(W, budget_s):
    """The plain C++ oracle (float32, -O3, no intrinsics) at 1 thread and at
    every host thread, scaled by packed bytes to the workload's step."""
    from oracle import cref
    mats, step_bytes = W.cpu_mats()
    nthreads = cref.hardware_threads()
    sample_bytes = sum(p.size for p, _ in mats)
    out = {}
    for th in (1, nthreads):
        rate, passes = cpu_gemv_rate(W.fmt, mats, budget_s / 2, th)
        out[th] = (rate, passes)
    to_unit = (lambda r: r / step_bytes * W.units_per_step) if W.unit == "tok/s" else (lambda r: r / 1e9)
    desc = (f"{len(mats)} matrices, {sample_bytes / 1e6:.0f} MB packed ({W.name}: "
            + ("layer 0's q/k/v, o, gate/up, down and 1/16 of the LM head" if W.name == "dense8b" else "the matrix")
            + "), scaled by bytes to the step; C++ oracle float32 dequant-GEMV, guided row split")
    return {"value": round(to_unit(out[nthreads][0]), 6), "unit": W.unit, "cores": nthreads, "kind": "oracle",
            "sample": desc, "passes": out[nthreads][1],
            "single_thread": {"value": round(to_unit(out[1][0]), 6), "cores": 1, "passes": out[1][1]}}


def cpu_baseline_moe(W, budget_s):
    v, sample = W.oracle_sample(budget_s=budget_s)
    return {"value": round(v, 6), "unit": W.unit, "cores": os.cpu_count(), "kind": "oracle", "sample": sample}


# ------------------------------------------------------------------ timing
def graph_of(torch, stream, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn(stream)
    return g


def time_replays(torch, stream, replay, steps):
    """Mean over `steps` back-to-back replays bracketed by one event pair,
    plus the median and minimum of `steps` individually timed replays."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            replay()
        e1.record(stream)
    e1.synchronize()
    mean = e0.elapsed_time(e1) / steps
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in pairs:
            a.record(stream)
            replay()
            b.record(stream)
    torch.cuda.synchronize()
    per = sorted(a.elapsed_time(b) for a, b in pairs)
    return mean, statistics.median(per), per[0]


def kernel_times(torch, W, stream, reps=3):
    """Per-launch time of each kernel of the step, in the regime the step runs
    it: a CUDA graph of N back-to-back launches of that kernel alone (distinct
    weights, programmatic dependent launch as in the step), CUDA events
    around `reps` replays; ms per launch."""
    out = {}
    for name in W.kernel_bytes:
        fn, n = W.kernel_bench(name)
        g = graph_of(torch, stream, fn)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
        mean, _, _ = time_replays(torch, stream, g.replay, reps)
        out[name] = mean / n
        del g
    return out


def roofline(W, ktimes, step_ms, peak, peak_kind):
    if not ktimes:
        return None
    dom = max(ktimes, key=lambda k: ktimes[k] * W.launches[k])
    ach = W.kernel_bytes[dom] / (ktimes[dom] * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get((W.name, dom))
    total = sum(ktimes[k] * W.launches[k] for k in ktimes)
    return {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
            "frac": round(ach / peak, 4), "peak_kind": peak_kind + " copy bandwidth",
            "traffic": tr[0] if tr else None, "traffic_source": tr[1] if tr else None,
            "avg_launch_us": round(ktimes[dom] * 1e3, 3), "bytes_per_launch": W.kernel_bytes[dom],
            "time_source": "graph of back-to-back launches of this kernel alone (distinct weights, PDL as in the "
                           "step), CUDA events around the replays",
            "kernels_us": {k: round(v * 1e3, 3) for k, v in ktimes.items()},
            "launches_per_step": W.launches,
            "sum_of_kernels_over_step": round(total / step_ms, 3)}


def make_workload(epq, dev, fmt, args, name=None, ntok=None, attn_ctx=-1, expert_fmt=None, down_fmt=None):
    name = name or args.workload
    if attn_ctx == -1:
        attn_ctx = args.attn_ctx
    if name == "moe_decode":
        ef = expert_fmt if expert_fmt is not None else (epq.FORMATS[args.expert_fmt] if args.expert_fmt else None)
        df = down_fmt if down_fmt is not None else (epq.FORMATS[args.down_fmt] if args.down_fmt else None)
        return MoEDecodeWorkload(epq, dev, fmt, layers=args.layers, attn_ctx=attn_ctx, expert_fmt=ef, down_fmt=df)
    if name == "moe_layer":
        return MoELayerWorkload(epq, dev, fmt, ntok=ntok or args.ntok)
    if name == "gemv4096":
        return Gemv4096Workload(epq, dev, fmt, nvec=args.nvec)
    if name == "dense8b":
        return DenseDecodeWorkload(epq, dev, fmt, nvec=args.nvec, layers=args.layers, chain=args.chain,
                                   attn_ctx=attn_ctx)
    raise SystemExit(f"unknown workload {name}")


def measure_workload(torch, epq, W, stream, steps, warmup, no_graph=False, clk=None):
    """Warm, capture and time one workload; returns a dict of measurements."""
    with torch.cuda.stream(stream):
        W.step(stream)
    stream.synchronize()
    assert epq.epq_device_error() == 0, "device-side wait timed out during warm-up"
    if no_graph:
        replay = lambda: W.step(stream)
    else:
        g = graph_of(torch, stream, W.step)
        replay = g.replay
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            replay()
    torch.cuda.synchronize()
    mean, med, mn = time_replays(torch, stream, replay, steps)
    return {"ms": mean, "ms_median": med, "ms_min": mn}


def e2e_measure(torch, W, stream, steps, no_graph):
    """Same step with pinned host input copied in and the result read back
    inside the timed region."""
    x_host = W.x.cpu().pin_memory()
    res_dev = W.out if hasattr(W, "out") else W.model.logits
    out_host = torch.empty(res_dev.shape, dtype=res_dev.dtype).pin_memory()
    x_dev = torch.empty_like(W.x)
    out_arg = res_dev if hasattr(W, "out") else None
    if no_graph:
        run = lambda: W.step(stream, x=x_dev, out=out_arg)
    else:
        g2 = graph_of(torch, stream, lambda s: W.step(s, x=x_dev, out=out_arg))
        run = g2.replay

    def one():
        x_dev.copy_(x_host, non_blocking=True)
        run()
        out_host.copy_(res_dev, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            one()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    n = max(1, min(steps, 5))
    with torch.cuda.stream(stream):
        e2.record(stream)
        for _ in range(n):
            one()
        e3.record(stream)
    e3.synchronize()
    return e2.elapsed_time(e3) / n, x_host.numel() * 4, out_host.numel() * 4


def eff_gbs(W, value_per_gpu):
    return W.bytes_per_token * value_per_gpu / 1e9 if W.unit == "tok/s" else value_per_gpu


def sub_object(torch, epq, W, stream, args, peak, peak_kind):
    """A compact measurement of one more workload for the headline line."""
    steps = max(5, min(args.steps, 10))
    m = measure_workload(torch, epq, W, stream, steps, 3)
    value = W.units_per_step / (m["ms"] * 1e-3)
    kt = kernel_times(torch, W, stream, reps=2)
    g = eff_gbs(W, value)
    obj = {"workload": W.config()["workload"], "value": round(value, 3), "unit": W.unit,
           "ms_per_step": round(m["ms"], 4), "ms_per_step_median": round(m["ms_median"], 4),
           "ms_per_step_min": round(m["ms_min"], 4), "steps": steps,
           "effective_weight_gbs": round(g, 1), "pct_of_measured_hbm": round(100 * g / peak, 2),
           "roofline": roofline(W, kt, m["ms"], peak, peak_kind), "config": W.config()}
    if hasattr(W, "extra"):
        obj.update(W.extra(value))
    if hasattr(W, "routing_report"):
        obj["routing"] = W.routing_report(stream)
    obj["device_error"] = epq.epq_device_error()
    return obj


def run_epq(args):
    import torch
    import moe_experts_gb300 as epq
    from moe_experts_gb300 import build as _build

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    _build.build()
    epq.load()
    if args.gemv_engine is not None:
        epq.epq_set_tuning(epq.EPQ_TUNE_GEMV_ENGINE, args.gemv_engine)
    for kv in args.tune:
        name, value = kv.split("=")
        if epq.epq_set_tuning(getattr(epq, "EPQ_TUNE_" + name.upper()), int(value)) < 0:
            raise SystemExit(f"--tune {kv}: value out of range")
    fmt = epq.FORMATS[args.fmt]
    W = make_workload(epq, dev, fmt, args)
    stream = torch.cuda.Stream(device=dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm + capture outside the clock record
    with torch.cuda.stream(stream):
        W.step(stream)
    stream.synchronize()
    assert epq.epq_device_error() == 0, "device-side wait timed out during warm-up"
    if args.no_graph:
        replay = lambda: W.step(stream)
    else:
        g = graph_of(torch, stream, W.step)
        replay = g.replay
    t_warm = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            replay()
    torch.cuda.synchronize()
    t_warm = (time.perf_counter() - t_warm) / max(3, args.warmup)
    # the clock record spans ~0.6 s of untimed back-to-back replays on each
    # side of the timed ones, so that its samples see the GPU under the load
    # of the timed region
    n_load = int(min(5000, max(1, 0.6 / max(t_warm, 1e-6))))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.mark_start()
        with torch.cuda.stream(stream):
            for _ in range(n_load):
                replay()
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # replays and events on one stream
            e0.record(stream)
            for _ in range(args.steps):
                replay()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(n_load):
                replay()
        torch.cuda.synchronize()
        clk.mark_end()
        barrier()
        clocks = clk.summary()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    # the same replays timed one by one (median and minimum)
    _, ms_med, ms_min = time_replays(torch, stream, replay, args.steps)
    ktimes = kernel_times(torch, W, stream) if not args.no_graph else {}
    err = epq.epq_device_error()
    e2e_ms, h2d, d2h = e2e_measure(torch, W, stream, args.steps, args.no_graph)
    e2e_ms = max_over_ranks(e2e_ms, dev)

    value = job_rate(W.units_per_step, ws, ms)
    peak, peak_kind = measured_peaks()
    g_eff = eff_gbs(W, value / ws)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": W.unit, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "ms_per_step_median": round(ms_med, 4),
        "ms_per_step_min": round(ms_min, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "q4k weights / f32 activations / f32 accumulate", "data": "synthetic",
        "config": {**W.config(), "parallelism": f"replicas{ws}" if ws > 1 else "single"},
        "effective_weight_gbs": round(g_eff, 1),
        "pct_of_measured_hbm": round(100 * g_eff / peak, 2),
        "pct_of_nominal_8tbs": round(100 * g_eff / NOMINAL_HBM_GBS, 2),
        "roofline": roofline(W, ktimes, ms, peak, peak_kind), "clocks": clocks,
        "gpu_launches": W.kernels_per_step * args.steps,
        "e2e": {"value": round(job_rate(W.units_per_step, ws, e2e_ms), 3), "unit": W.unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "device_error": err,
    }
    if hasattr(W, "extra"):
        line.update(W.extra(value / ws))
    if hasattr(W, "routing_report") and rank == 0:
        line["routing"] = W.routing_report(stream)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        if hasattr(W, "cpu_mats"):
            line["cpu_baseline"] = cpu_baseline_gemv(W, args.cpu_budget)
        else:
            line["cpu_baseline"] = cpu_baseline_moe(W, args.cpu_budget)
    if rank == 0 and ws == 1 and args.workload == "dense8b" and not (args.no_sub or args.chain or args.no_graph):
        # the other configurations, measured in the same run (compact)
        del g, replay, W
        torch.cuda.empty_cache()
        subs = {}
        Q2K, Q6K = epq.EPQ_Q2_K, epq.EPQ_Q6_K
        for key, name, ntok, ctx, wfmt, ef, df, nv in (
                ("gemv4096", "gemv4096", None, None, fmt, None, None, 1),
                ("gemv4096_q2k", "gemv4096", None, None, Q2K, None, None, 1),
                ("gemv4096_q6k", "gemv4096", None, None, Q6K, None, None, 1),
                ("moe_layer_1tok", "moe_layer", 1, None, fmt, None, None, 1),
                ("moe_layer_8tok", "moe_layer", 8, None, fmt, None, None, 1),
                ("moe_decode", "moe_decode", None, None, fmt, None, None, 1),
                ("moe_decode_q2k_experts", "moe_decode", None, None, fmt, Q2K, None, 1),
                ("moe_decode_q6k_down", "moe_decode", None, None, fmt, None, Q6K, 1),
                ("dense8b_attn1024", "dense8b", None, 1024, fmt, None, None, 1),
                ("moe_decode_attn1024", "moe_decode", None, 1024, fmt, None, None, 1),
                ("dense8b_verify2", "dense8b", None, None, fmt, None, None, 2),
                ("dense8b_verify8", "dense8b", None, None, fmt, None, None, 8)):
            Wk = make_workload(epq, dev, wfmt, argparse.Namespace(**{**vars(args), "layers": None, "nvec": nv}),
                               name=name, ntok=ntok, attn_ctx=ctx, expert_fmt=ef, down_fmt=df)
            subs[key] = sub_object(torch, epq, Wk, stream, args, peak, peak_kind)
            del Wk
            torch.cuda.empty_cache()
        line["sub_workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle, timed on the host cores: each step is one bounded sample of
    the same workload (the other ranks of a multi-GPU launch exit without
    work).  Inputs are drawn with the same generators and packed by the
    oracle itself."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    import torch
    from oracle import cref
    from synthetic import workloads as wl
    fmt = {"Q8_0": 0, "Q4_0": 1, "Q4_1": 2, "Q4_K": 3, "Q2_K": 4, "Q6_K": 5}[args.fmt]
    nthreads = cref.hardware_threads()
    t_all = time.perf_counter()
    if args.workload in ("dense8b", "gemv4096"):
        pack = lambda Wf: cref.quantize(fmt, Wf.numpy(), threads=nthreads)
        rb = lambda cols: cref.row_bytes(fmt, cols)
        if args.workload == "dense8b":
            c = wl.DenseDecode()
            H, nq, nkv, I, V = c.hidden, c.q_rows, c.kv_rows, c.inter, c.vocab
            mats = [(np.concatenate([pack(wl.weight("dense8b", 0, 0, nq, H, "cpu")),
                                     pack(wl.weight("dense8b", 0, 1, nkv, H, "cpu")),
                                     pack(wl.weight("dense8b", 0, 2, nkv, H, "cpu"))]), H),
                    (pack(wl.weight("dense8b", 0, 3, H, nq, "cpu")), nq),
                    (np.concatenate([pack(wl.weight("dense8b", 0, 4, I, H, "cpu")),
                                     pack(wl.weight("dense8b", 0, 5, I, H, "cpu"))]), H),
                    (pack(wl.weight("dense8b", 0, 6, H, I, "cpu")), I),
                    (pack(wl.weight("dense8b", 0, 7, V // 16, H, "cpu")), H)]
            step_bytes = c.layers * ((nq + 2 * nkv) * rb(H) + H * rb(nq) + 2 * I * rb(H) + H * rb(I)) + V * rb(H)
            unit, units = "tok/s", float(args.nvec)
            cfg = {"workload": "dense8b_decode_q4k", "layers": c.layers, "hidden": H, "inter": I, "vocab": V,
                   "nvec": args.nvec, "batch": 1}
            desc = "layer 0's q/k/v, o, gate/up, down and 1/16 of the LM head, scaled by bytes to the full step"
        else:
            packed = pack(wl.weight("gemv4096", 0, 0, 4096, 4096, "cpu"))
            mats = [(packed, 4096)]
            step_bytes = packed.size
            unit, units = "GB/s", packed.size / 1e9
            cfg = {"workload": f"gemv4096_{FMT_TAG[fmt]}", "rows": 4096, "cols": 4096, "nvec": args.nvec, "batch": 1}
            desc = "the 4096x4096 matrix, one GEMV per step"
        sample_bytes = sum(p.size for p, _ in mats)
        xs = [np.random.default_rng(3).standard_normal((args.nvec, cols)).astype(np.float32) for _, cols in mats]
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            for (p, cols), x in zip(mats, xs):
                cref.gemv_f32(fmt, p, x, cols, threads=nthreads)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        t_step = statistics.mean(times)
        value = units / (t_step * step_bytes / sample_bytes) if unit == "tok/s" else sample_bytes / t_step / 1e9
        ms_sample = 1e3 * t_step
        dtype = "f32 (C++ oracle)"
        sample = (f"{desc}; {sample_bytes / 1e6:.0f} MB packed per step, C++ oracle float32 dequant-GEMV, "
                  f"{nthreads} threads, guided row split")
    else:
        import moe_experts_gb300 as epq
        from moe_experts_gb300 import build as _build
        _build.build()
        epq.load()
        dev = torch.device(f"cuda:{local}")
        efmt = epq.FORMATS[args.fmt]
        if args.workload == "moe_decode":
            W = MoEDecodeWorkload(epq, dev, efmt, layers=1,
                                  expert_fmt=epq.FORMATS[args.expert_fmt] if args.expert_fmt else None,
                                  down_fmt=epq.FORMATS[args.down_fmt] if args.down_fmt else None)
            W.cfg = wl.MoEDecode()
        else:
            W = MoELayerWorkload(epq, dev, efmt, ntok=args.ntok, replicas=1)
        unit, cfg, dtype = W.unit, W.config(), "f64 (numpy oracle)"
        per_step = args.cpu_budget / max(1, args.steps + args.warmup)
        vals, times = [], []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            v, sample = W.oracle_sample(budget_s=per_step)
            if i >= args.warmup:
                vals.append(v)
                times.append(time.perf_counter() - t0)
        value = statistics.mean(vals)
        ms_sample = 1e3 * statistics.mean(times)
        nthreads = os.cpu_count()
    wall = time.perf_counter() - t_all
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_sample, 3),
            "ms_per_step_meaning": "wall time of one bounded sample step (what each timed step ran)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="epq", choices=["epq", "reference"])
    ap.add_argument("--workload", default="dense8b", choices=["dense8b", "gemv4096", "moe_decode", "moe_layer"])
    ap.add_argument("--ntok", type=int, default=1, help="tokens per MoE layer forward (moe_layer)")
    ap.add_argument("--chain", action="store_true", help="dense step as one epq_gemv_chain launch")
    ap.add_argument("--fmt", default="Q4_K", choices=["Q8_0", "Q4_0", "Q4_1", "Q4_K", "Q2_K", "Q6_K"])
    ap.add_argument("--expert-fmt", default=None, choices=["Q8_0", "Q4_0", "Q4_1", "Q4_K", "Q2_K", "Q6_K"],
                    help="moe_decode: format of the experts (default --fmt)")
    ap.add_argument("--down-fmt", default=None, choices=["Q8_0", "Q4_0", "Q4_1", "Q4_K", "Q2_K", "Q6_K"],
                    help="moe_decode: format of the experts' down projections (a mixed recipe)")
    ap.add_argument("--nvec", type=int, default=1)
    ap.add_argument("--attn-ctx", type=int, default=None,
                    help="decode with KV-cache attention over this many cached positions (dense8b, moe_decode)")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (smaller cases)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the other workloads' sub-objects")
    ap.add_argument("--no-graph", action="store_true", help="launch each step directly (no CUDA graph)")
    ap.add_argument("--gemv-engine", type=int, default=None,
                    help="EPQ_TUNE_GEMV_ENGINE for this run (0 automatic, 1 CUDA cores, 2 tensor cores, "
                         "3 block-diagonal tensor-core engine for Q4_K, 4 vector-column engine for 2+ vectors)")
    ap.add_argument("--tune", action="append", default=[], metavar="NAME=VALUE",
                    help="an epq_set_tuning key for this run, e.g. VN_CLUSTER=4 (EPQ_TUNE_ prefix dropped)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_epq(args)


if __name__ == "__main__":
    main()
