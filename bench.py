"""Benchmark of the block-quantized decode path on GB300.

Default workload (the headline): the full dense 8B-class decode step with
Q4_K weights -- 32 layers (q 4096x4096, k/v 1024x4096, o 4096x4096, gate/up
2x14336x4096 with SwiGLU, down 4096x14336, weightless RMS pre-norms, a
one-token-context attention stand-in) plus the 128256x4096 LM head, batch 1
(--nvec 2/4/8 for speculative-verify columns).  One "step" = one token
through all 129 dequant-GEMVs, replayed from one CUDA graph.  4.2 GB of
packed weights stay resident and every step streams all of them, far beyond
the 129 MB L2, so no flush is needed.

Other workloads (--workload): moe_decode (40 MoE layers, hidden 2048, 256
experts of gate/up 512x2048 + down 2048x512, top-8 + shared expert, Zipf(1.1)
routing, a 64-token decode run per step); moe_layer (one MoE layer of hidden
4096 with 512 experts of gate/up 2x1024x4096 + down 4096x1024, top-4 + shared
expert, --ntok 1 or 8 tokens per forward; value = effective weight GB/s).
--chain runs the dense step as one epq_gemv_chain launch instead of one
launch per matrix.

The JSON line carries: value (tok/s for decode workloads, GB/s otherwise),
roofline of the dominant kernel (live CUDA-event pairs inside the graph),
e2e (host buffers, H2D + D2H inside the timed region), clocks sampled
during the timed region, gpu_launches, and the CPU baseline (the oracle on
a bounded sample).  --impl reference times the oracle itself.
"""
from __future__ import annotations

import argparse
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
    ("dense8b", "gemv_gateup"): (66_333_184, "profiles/gemv_tc_gateup_q4k_full.md"),
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
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
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

    def summary(self):
        sm, smax, reasons = [], [], set()
        try:
            for line in open(self.path):
                f = [v.strip() for v in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    smax.append(float(f[2]))
                except ValueError:
                    continue
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except Exception:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


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


class MoEDecodeWorkload(Workload):
    name = "moe_decode"
    unit = "tok/s"

    def __init__(self, epq, dev, fmt, layers=None):
        from synthetic import workloads as wl
        self.cfg = c = wl.MoEDecode() if layers is None else wl.MoEDecode(layers=layers)
        self.fmt, self.dev, self.epq = fmt, dev, epq
        H, I, E = c.hidden, c.inter, c.n_experts
        rbH, rbI = epq.epq_row_bytes(fmt, H), epq.epq_row_bytes(fmt, I)
        import torch
        self.layers = []
        for l in range(c.layers):
            wqkv = torch.empty((3 * H, rbH), dtype=torch.uint8, device=dev)
            for t in range(3):
                epq.epq_quantize(fmt, wl.weight("moe_decode", l, t, H, H, dev), blocks=wqkv[t * H:(t + 1) * H])
            wo = epq.epq_quantize(fmt, wl.weight("moe_decode", l, 3, H, H, dev))
            R, bias = wl.moe_router("moe_decode", l, E, H, dev, c.zipf_s)
            gu = torch.empty((E, 2 * I, rbH), dtype=torch.uint8, device=dev)
            dn = torch.empty((E, H, rbI), dtype=torch.uint8, device=dev)
            for e0 in range(0, E, 64):
                n = min(64, E - e0)
                Wg = wl.weight("moe_decode", l, 10, n * 2 * I, H, dev, expert=e0)
                epq.epq_quantize(fmt, Wg, blocks=gu[e0:e0 + n].view(n * 2 * I, rbH))
                Wd = wl.weight("moe_decode", l, 11, n * H, I, dev, expert=e0)
                epq.epq_quantize(fmt, Wd, blocks=dn[e0:e0 + n].view(n * H, rbI))
                del Wg, Wd
            sgu = epq.epq_quantize(fmt, wl.weight("moe_decode", l, 12, 2 * I, H, dev))
            sdn = epq.epq_quantize(fmt, wl.weight("moe_decode", l, 13, H, I, dev))
            layer = epq.MoELayer(fmt, R, gu, dn, router_bias=bias, shared_gate_up=sgu, shared_down=sdn)
            self.layers.append((wqkv, wo, layer))
        torch.cuda.synchronize()
        from moe_experts_gb300.decode import MoEDecoder
        self.model = MoEDecoder(c, fmt, self.layers, dev)
        self.T = c.tokens
        self.x = wl.activations("moe_decode", self.T, H, dev)
        self.out = torch.empty((self.T, H), dtype=torch.float32, device=dev)
        self.units_per_step = float(self.T)
        self.bytes_per_token = c.layers * (4 * H * rbH + E * H * 4 + (c.topk + 1) * (2 * I * rbH + H * rbI))
        self.kernels_per_step = self.T * c.layers * 5
        # dominant-kernel candidates: name -> (algorithmic bytes per launch, launches per step)
        self.kernel_bytes = {
            "gemv_qkv": 3 * H * rbH + 4 * (H + 3 * H),
            "gemv_o": H * rbH + 4 * (H + 2 * H),
            "moe_router": E * H * 4 + 4 * H,
            "moe_gateup": (c.topk + 1) * 2 * I * rbH + 4 * (H + (c.topk + 1) * I),
            "moe_down": (c.topk + 1) * H * rbI + 4 * ((c.topk + 1) * I + 2 * H),
        }

    def config(self):
        c = self.cfg
        return {"workload": "moe_decode_q4k", "layers": c.layers, "hidden": c.hidden, "experts": c.n_experts,
                "inter": c.inter, "topk": c.topk, "shared_experts": 1, "tokens_per_step": c.tokens, "batch": 1,
                "router": "fp32 zipf(1.1)", "weights_resident_gb": round(self.resident_gb(), 2),
                "bytes_per_token": self.bytes_per_token, "l2": "inputs larger than L2 (1.1 GB/token)"}

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
            self.model.token(x[t:t + 1], out[t:t + 1], stream=stream, timers=timers if t < 64 else None)

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
                o = oracle.expert_forward_f64(self.fmt, gu_all[int(e)].cpu().numpy(), dn_all[int(e)].cpu().numpy(),
                                              H, I, xin[0])[0]
                y += w[0, k] * o
            o = oracle.expert_forward_f64(self.fmt, mw.shared_gate_up, mw.shared_down, H, I, xin[0])[0]
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

    def __init__(self, epq, dev, fmt, nvec=1, layers=None, chain=False):
        import torch
        from synthetic import workloads as wl
        self.cfg = c = wl.DenseDecode() if layers is None else wl.DenseDecode(layers=layers)
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
        self.model = DenseDecoder(c, fmt, self.layers, head, dev, nvec=nvec, chain=chain)
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
        self.kernels_per_step = 1 if chain else c.layers * 4 + 1
        if chain:  # the one launch is the dominant (and only) kernel
            self.kernel_bytes = {"gemv_chain": wbytes + 4 * nvec * (c.layers * (4 * H + 2 * c.inter + nq + 2 * nkv
                                                                                 + H) + H + c.vocab)}
        else:
            self.kernel_bytes = {
                "gemv_qkv": (nq + 2 * nkv) * rbH + 4 * nvec * (H + nq + 2 * nkv),
                "gemv_o": H * epq.epq_row_bytes(fmt, nq) + 4 * nvec * (nkv + 2 * H),
                "gemv_gateup": 2 * c.inter * rbH + 4 * nvec * (H + c.inter),
                "gemv_down": H * rbI + 4 * nvec * (c.inter + 2 * H),
            }

    def config(self):
        c = self.cfg
        return {"workload": f"dense8b_decode_{'q4k' if self.fmt == 3 else self.fmt}", "layers": c.layers,
                "launch": "one epq_gemv_chain launch per step" if self.chain else "one launch per matrix",
                "hidden": c.hidden, "inter": c.inter, "heads": c.heads, "kv_heads": c.kv_heads, "vocab": c.vocab,
                "nvec": self.nvec, "batch": 1, "weight_bytes_per_step": self.weight_bytes_per_step,
                "l2": "inputs larger than L2 (4.2 GB/step)"}

    def step(self, stream, x=None, out=None, timers=None):
        self.model.step(self.x if x is None else x, stream=stream, timers=timers)

    def oracle_sample(self, budget_s=20.0):
        import numpy as np
        import oracle
        c = self.cfg
        H = c.hidden
        x = self.x.cpu().numpy().astype(np.float64)
        t0 = time.perf_counter()
        done = 0
        nbytes = 0
        for wqkv, wo, wgu, wd in self.layers:
            for w, cols in ((wqkv, H), (wgu, H)):
                p = w.cpu().numpy()
                oracle.gemv_f64(self.fmt, p, x, cols)
                nbytes += p.size
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        # scale by bytes: the sample covered qkv + gate/up of `done` layers
        rate = nbytes / dt
        return rate / (self.full_step_bytes / self.nvec), \
            f"{done} layers' qkv+gate/up GEMVs (oracle, float64), scaled by bytes to the full step"


# ------------------------------------------------------------------ timing
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
    fmt = epq.FORMATS[args.fmt]
    if args.workload == "moe_decode":
        W = MoEDecodeWorkload(epq, dev, fmt, layers=args.layers)
    elif args.workload == "moe_layer":
        W = MoELayerWorkload(epq, dev, fmt, ntok=args.ntok)
    elif args.workload == "dense8b":
        W = DenseDecodeWorkload(epq, dev, fmt, nvec=args.nvec, layers=args.layers, chain=args.chain)
    else:
        raise SystemExit(f"unknown workload {args.workload}")

    stream = torch.cuda.Stream(device=dev)
    # warm the kernels (sets smem attributes) outside capture
    with torch.cuda.stream(stream):
        W.step(stream)
    stream.synchronize()
    assert epq.epq_device_error() == 0, "device-side wait timed out during warm-up"

    # The timed steps carry no instrumentation.  Per-kernel durations come
    # from a second capture of the same step with CUDA event pairs around the
    # kernels of its first layer, replayed after the timed region.
    timers = Timers(torch, W)
    if args.no_graph:  # direct launches (for profilers that do not follow graph replays)
        def replay():
            W.step(stream)

        def replay_timed():
            W.step(stream, timers=timers)
    else:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            W.step(stream)
        replay = g.replay
        gt = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gt, stream=stream):
            W.step(stream, timers=timers)
        replay_timed = gt.replay
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            replay()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):  # replays and events on one stream
            e0.record(stream)
            for _ in range(args.steps):
                replay()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        barrier()
    ms = e0.elapsed_time(e1) / args.steps
    with torch.cuda.stream(stream):
        for _ in range(max(1, min(args.steps, 5))):
            replay_timed()
    torch.cuda.synchronize()
    kernel_ms = timers.averages()
    clocks = clk.summary()
    err = epq.epq_device_error()
    ms = max_over_ranks(ms, dev)

    # ---- end to end: host (pinned) inputs in, results back to host, per step
    x_host = W.x.cpu().pin_memory()
    out_dev = torch.empty_like(W.out if hasattr(W, "out") else W.model.logits)
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    x_dev = torch.empty_like(W.x)
    if args.no_graph:
        class _Direct:
            def replay(self):
                W.step(stream, x=x_dev, out=out_dev if hasattr(W, "out") else None)
        g2 = _Direct()
    else:
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            W.step(stream, x=x_dev, out=out_dev if hasattr(W, "out") else None)
    res_src = out_dev if hasattr(W, "out") else W.model.logits
    with torch.cuda.stream(stream):
        for _ in range(2):
            x_dev.copy_(x_host, non_blocking=True)
            g2.replay()
            out_host.copy_(res_src, non_blocking=True)
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, min(args.steps, 5))
    barrier()
    e2.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(n_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            g2.replay()
            out_host.copy_(res_src, non_blocking=True)
    e3.record(stream)
    e3.synchronize()
    e2e_ms = max_over_ranks(e2.elapsed_time(e3) / n_e2e, dev)

    value = job_rate(W.units_per_step, ws, ms)
    peak, peak_kind = measured_peaks()
    # dominant kernel: largest total time per step
    launches = {k: W.kernels_per_step // len(W.kernel_bytes) for k in W.kernel_bytes}
    dom = max(kernel_ms, key=lambda k: kernel_ms[k] * launches[k]) if kernel_ms else None
    roof = None
    if dom:
        ach = W.kernel_bytes[dom] / (kernel_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_kind": peak_kind + " copy bandwidth",
                "traffic": NCU_TRAFFIC[(W.name, dom)][0] if (W.name, dom) in NCU_TRAFFIC else None,
                "traffic_source": NCU_TRAFFIC[(W.name, dom)][1] if (W.name, dom) in NCU_TRAFFIC else None,
                "avg_launch_us": round(kernel_ms[dom] * 1e3, 3),
                "bytes_per_launch": W.kernel_bytes[dom],
                "all_kernels_us": {k: round(v * 1e3, 3) for k, v in kernel_ms.items()}}
    eff_gbs = W.bytes_per_token * (value / ws) / 1e9 if W.unit == "tok/s" else value / ws
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": W.unit, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "q4k weights / f32 activations / f32 accumulate", "data": "synthetic",
        "config": {**W.config(), "parallelism": f"replicas{ws}" if ws > 1 else "single"},
        "effective_weight_gbs": round(eff_gbs, 1) if eff_gbs else None,
        "pct_of_measured_hbm": round(100 * eff_gbs / peak, 2) if eff_gbs else None,
        "pct_of_nominal_8tbs": round(100 * eff_gbs / NOMINAL_HBM_GBS, 2) if eff_gbs else None,
        "roofline": roof, "clocks": clocks, "gpu_launches": W.kernels_per_step * args.steps,
        "e2e": {"value": round(job_rate(W.units_per_step, ws, e2e_ms), 3), "unit": W.unit,
                "h2d_bytes_per_step": x_host.numel() * 4, "d2h_bytes_per_step": out_host.numel() * 4},
        "device_error": err,
    }
    if hasattr(W, "extra"):
        line.update(W.extra(value / ws))
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, sample = W.oracle_sample(budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": W.unit, "cores": os.cpu_count(), "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class Timers:
    """CUDA event pairs recorded (as graph nodes) around each kernel of
    layer 0 for every token of the step; averaged after the timed region."""

    def __init__(self, torch, W):
        self.torch = torch
        self.pairs = {}
        self.names = list(W.kernel_bytes)

    def pair(self, name):
        t = self.torch
        a = t.cuda.Event(enable_timing=True, external=True)
        b = t.cuda.Event(enable_timing=True, external=True)
        self.pairs.setdefault(name, []).append((a, b))
        return a, b

    def averages(self):
        out = {}
        for k, ps in self.pairs.items():
            v = [a.elapsed_time(b) for a, b in ps]
            out[k] = sum(v) / len(v)
        return out


def run_reference(args):
    """The oracle, timed on the host cores, on a bounded sample of the same
    workload (the other ranks of a multi-GPU launch exit without work)."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import torch
    import moe_experts_gb300 as epq
    from moe_experts_gb300 import build as _build
    _build.build()
    epq.load()
    dev = torch.device(f"cuda:{local}")
    fmt = epq.FORMATS[args.fmt]
    # the reference arm only needs the packed weights of the sampled layers
    if args.workload == "moe_decode":
        W = MoEDecodeWorkload(epq, dev, fmt, layers=max(1, args.ref_layers))
        W.cfg = __import__("synthetic.workloads", fromlist=["MoEDecode"]).MoEDecode()
    elif args.workload == "moe_layer":
        W = MoELayerWorkload(epq, dev, fmt, ntok=args.ntok, replicas=1)
    else:
        W = DenseDecodeWorkload(epq, dev, fmt, nvec=args.nvec, layers=max(1, args.ref_layers))
    per_step = args.cpu_budget / max(1, args.steps + args.warmup)
    vals = []
    t_all = time.perf_counter()
    for i in range(args.warmup + args.steps):
        v, sample = W.oracle_sample(budget_s=per_step)
        if i >= args.warmup:
            vals.append(v)
    dt = time.perf_counter() - t_all
    value = statistics.mean(vals)
    ms = 1e3 * W.units_per_step / value
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": W.unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3) if ms else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": W.config(),
            "cpu_baseline": {"value": round(value, 6), "unit": W.unit, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": W.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(dt, 1)}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="epq", choices=["epq", "reference"])
    ap.add_argument("--workload", default="dense8b", choices=["dense8b", "moe_decode", "moe_layer"])
    ap.add_argument("--ntok", type=int, default=1, help="tokens per MoE layer forward (moe_layer)")
    ap.add_argument("--chain", action="store_true", help="dense step as one epq_gemv_chain launch")
    ap.add_argument("--fmt", default="Q4_K", choices=["Q8_0", "Q4_0", "Q4_1", "Q4_K"])
    ap.add_argument("--nvec", type=int, default=1)
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (smaller cases)")
    ap.add_argument("--ref-layers", type=int, default=2)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each step directly (no CUDA graph)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_epq(args)


if __name__ == "__main__":
    main()
