"""GPU parity of epq_gemv_chain (a chain of dependent Q4_K GEMVs in one
persistent launch) against the float64 oracle, stage by stage.

Each op writes its own buffer, so after the chain every op's inputs (earlier
ops' outputs) and output are available: the oracle recomputes the op from the
chain's own inputs (the stage-wise method of [E] "正確性") and the op must be
within the GEMV bound 1e-4 * sum_j |w_ij x_j| (plus |residual|; SwiGLU
outputs within the propagated bound).  The chain is a small dense decoder
(pre-norm, grouped-head attention over a one-token context, SwiGLU MLP) plus
an LM head, and one layer of the 8B-class decoder at full size (sampled).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

Q4K = oracle.Q4_K
TOL = 1e-4


def _expand_heads(v, hd, grp):
    """x of a grouped-head op: each hd-float head of v repeated grp times."""
    nh = v.shape[1] // hd
    return np.concatenate([np.tile(v[:, h * hd:(h + 1) * hd], (1, grp)) for h in range(nh)], axis=1)


def _within(y, ref, A, what):
    err = np.abs(y.astype(np.float64) - ref)
    lim = TOL * A + 1e-30
    assert (err <= lim).all(), f"{what}: worst ratio {(err / lim).max():.3g}"


class _Model:
    def __init__(self, epq, dev, nvec, L=2, H=1024, nq=1024, nkv=256, hd=64, I=2816, V=3000, seed=0,
                 full_check=True):
        self.epq, self.dev, self.nvec = epq, dev, nvec
        self.H, self.nq, self.nkv, self.hd, self.I, self.V, self.L = H, nq, nkv, hd, I, V, L
        self.grp = nq // nkv
        self.eps = 1e-5
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        # float32 weights stay on the device: the check packs its sampled rows with the oracle
        self.W, self.Wf = [], []
        for l in range(L):
            mats, fl = {}, {}
            for name, (r, c) in {"qkv": (nq + 2 * nkv, H), "o": (H, nq), "gu": (2 * I, H), "d": (H, I)}.items():
                fl[name] = synthetic.student_t((r, c), seed=seed * 100 + l * 10 + len(mats), device=dev)
                mats[name] = epq.epq_quantize(Q4K, fl[name])
            self.W.append(mats)
            self.Wf.append(fl)
        self.headf = synthetic.student_t((V, H), seed=seed * 100 + 99, device=dev)
        self.head = epq.epq_quantize(Q4K, self.headf)
        self.x = synthetic.normal((nvec, H), seed=seed + 7, device=dev)
        f = lambda n: torch.empty((nvec, n), dtype=torch.float32, device=dev)
        self.buf = [{"qkv": f(nq + 2 * nkv), "h1": f(H), "m": f(I), "h2": f(H)} for _ in range(L)]
        self.logits = f(V)
        self.ws = torch.zeros(epq.epq_gemv_chain_workspace_bytes(), dtype=torch.uint8, device=dev)

    def ops(self):
        e, H, nq, nkv = self.epq, self.H, self.nq, self.nkv
        ops = []
        h = self.x
        for l in range(self.L):
            W, B = self.W[l], self.buf[l]
            ops.append(e.gemv_op(W["qkv"], h, B["qkv"], nq + 2 * nkv, H, rms_prenorm=True, rms_eps=self.eps))
            ops.append(e.gemv_op(W["o"], B["qkv"][:, nq + nkv:], B["h1"], H, nq, residual=h,
                                 x_group=self.grp, x_head_dim=self.hd))
            ops.append(e.gemv_op(W["gu"], B["h1"], B["m"], 2 * self.I, H, swiglu=True, rms_prenorm=True,
                                 rms_eps=self.eps))
            ops.append(e.gemv_op(W["d"], B["m"], B["h2"], H, self.I, residual=B["h1"]))
            h = B["h2"]
        ops.append(e.gemv_op(self.head, h, self.logits, self.V, H, rms_prenorm=True, rms_eps=self.eps))
        return ops

    def run(self, stream=None):
        self.epq.epq_gemv_chain(Q4K, self.ops(), self.nvec, self.ws, stream=stream)

    def packed(self, blocks, wf, rows):
        """Oracle packing of the sampled rows (the GPU's packing must equal it)."""
        ix = torch.from_numpy(rows).to(self.dev)
        pk = oracle.quantize(Q4K, wf[ix].cpu().numpy())
        assert np.array_equal(pk, blocks[ix].cpu().numpy())
        return pk

    def check(self, rows_sample=None):
        """Every op against the oracle on the chain's own inputs."""
        cpu = lambda a: a.cpu().numpy()
        rng = np.random.default_rng(1)
        def pick(n):
            return np.arange(n) if rows_sample is None or n <= rows_sample else np.sort(
                rng.choice(n, rows_sample, replace=False))
        h = cpu(self.x).astype(np.float64)
        for l in range(self.L):
            W, B, Wf = self.W[l], self.buf[l], self.Wf[l]
            # qkv = W rms(h)
            r = pick(self.nq + 2 * self.nkv)
            pk = self.packed(W["qkv"], Wf["qkv"], r)
            xn = oracle.rmsnorm_f64(h, self.eps)
            _within(cpu(B["qkv"])[:, r], oracle.gemv_f64(Q4K, pk, xn, self.H), oracle.gemv_bound(Q4K, pk, xn, self.H),
                    f"layer {l} qkv")
            # h1 = h + Wo expand(v)
            v = cpu(B["qkv"])[:, self.nq + self.nkv:].astype(np.float64)
            xe = _expand_heads(v, self.hd, self.grp)
            r = pick(self.H)
            pk = self.packed(W["o"], Wf["o"], r)
            ref = h[:, r] + oracle.gemv_f64(Q4K, pk, xe, self.nq)
            _within(cpu(B["h1"])[:, r], ref, oracle.gemv_bound(Q4K, pk, xe, self.nq) + np.abs(h[:, r]),
                    f"layer {l} o")
            h1 = cpu(B["h1"]).astype(np.float64)
            # m = silu(Wg rms(h1)) * (Wu rms(h1))
            r = pick(self.I)
            rr = np.concatenate([r, r + self.I])
            pk = self.packed(W["gu"], Wf["gu"], rr)
            xn = oracle.rmsnorm_f64(h1, self.eps)
            y = oracle.gemv_f64(Q4K, pk, xn, self.H)
            A = oracle.gemv_bound(Q4K, pk, xn, self.H)
            n = len(r)
            g, u, Ag, Au = y[:, :n], y[:, n:], A[:, :n], A[:, n:]
            silu = g / (1 + np.exp(-g))
            bound = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(silu * u)
            err = np.abs(cpu(B["m"])[:, r] - silu * u)
            assert (err <= bound + 1e-30).all(), f"layer {l} gate/up: {(err / (bound + 1e-30)).max():.3g}"
            # h2 = h1 + Wd m
            m = cpu(B["m"]).astype(np.float64)
            r = pick(self.H)
            pk = self.packed(W["d"], Wf["d"], r)
            ref = h1[:, r] + oracle.gemv_f64(Q4K, pk, m, self.I)
            _within(cpu(B["h2"])[:, r], ref, oracle.gemv_bound(Q4K, pk, m, self.I) + np.abs(h1[:, r]),
                    f"layer {l} down")
            h = cpu(B["h2"]).astype(np.float64)
        r = pick(self.V)
        pk = self.packed(self.head, self.headf, r)
        xn = oracle.rmsnorm_f64(h, self.eps)
        _within(cpu(self.logits)[:, r], oracle.gemv_f64(Q4K, pk, xn, self.H), oracle.gemv_bound(Q4K, pk, xn, self.H),
                "head")


@pytest.mark.parametrize("nvec", [1, 2])
def test_chain_small_decoder(epq_lib, cuda_dev, nvec):
    m = _Model(epq_lib, cuda_dev, nvec)
    m.run()
    torch.cuda.synchronize()
    assert epq_lib.epq_device_error() == 0
    m.check()


def test_chain_deterministic_and_graph_replay(epq_lib, cuda_dev):
    """Repeated calls (workspace reused) and CUDA-graph replays give the same bits."""
    m = _Model(epq_lib, cuda_dev, 2, L=3, seed=3)
    m.run()
    ref = m.logits.clone()
    m.run()
    assert torch.equal(m.logits, ref)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.run(stream=s)
    for _ in range(2):
        m.logits.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(m.logits, ref)
    assert epq_lib.epq_device_error() == 0
    m.check()


def test_chain_full_size_layer(epq_lib, cuda_dev):
    """One layer of the 8B-class decoder (q 4096, k/v 1024, o 4096x4096,
    gate/up 2x14336, down 4096x14336) and the 128256-row LM head; 128 rows of
    every op checked against the oracle."""
    m = _Model(epq_lib, cuda_dev, 1, L=1, H=4096, nq=4096, nkv=1024, hd=128, I=14336, V=128256, seed=5)
    m.run()
    torch.cuda.synchronize()
    assert epq_lib.epq_device_error() == 0
    m.check(rows_sample=128)


def test_chain_argument_errors(epq_lib, cuda_dev):
    m = _Model(epq_lib, cuda_dev, 1, L=1, seed=9)
    ops = m.ops()
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv_chain(oracle.Q4_0, ops, 1, m.ws)                       # format
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv_chain(Q4K, ops, 3, m.ws)                               # nvec > 2
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv_chain(Q4K, ops, 1, m.ws[:16])                          # workspace too small
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv_chain(Q4K, [], 1, m.ws)                                # no ops
