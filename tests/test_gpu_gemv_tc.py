"""GPU parity of the tensor-core Q4_K dequant-GEMV engine against the float64
oracle, with the engine forced on for every shape (the automatic choice uses
it only for large matrices and for two or more vectors).

Bar (the accuracy target of the GEMV): |y_gpu - y_ref| <= 1e-4 * sum_j |deq(W)_ij x_j|
per row and vector.  Shapes cover one and several stages per CTA, ragged row
counts (rows not a multiple of the 8-row MMA block), every warp split of the
engine (1 to 16 warps per row block, 1 to 4 superblocks per warp, superblock
counts that do not divide evenly) and SwiGLU pairs.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4
Q4K = oracle.Q4_K


@pytest.fixture()
def tc_engine(epq_lib):
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, 2)
    yield epq_lib
    epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


def _check(y_gpu, y_ref, A, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    lim = TOL * A + 1e-30
    bad = np.argwhere(err > lim)
    assert bad.size == 0, f"{what}: {bad.shape[0]} outputs beyond bound, first {bad[:3].tolist()}, " \
                          f"worst ratio {(err / lim).max():.3g}"


SHAPES = [(1, 256), (7, 512), (9, 768), (33, 1024), (130, 4096), (257, 2048), (20, 14336), (1000, 768),
          (3, 1280), (1217, 4096), (40, 12288), (4000, 256), (2500, 2048), (17, 16384)]


@pytest.mark.parametrize("shape", SHAPES)
def test_tc_parity(tc_engine, cuda_dev, shape):
    rows, cols = shape
    for nvec in (1, 2, 3):
        seed = rows * 131 + cols + nvec
        W = synthetic.student_t((rows, cols), seed=seed).numpy()
        x = synthetic.normal((nvec, cols), seed=seed + 1).numpy()
        packed = oracle.quantize(Q4K, W)
        y = tc_engine.epq_gemv(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                               rows, cols).cpu().numpy()
        _check(y, oracle.gemv_f64(Q4K, packed, x, cols), oracle.gemv_bound(Q4K, packed, x, cols),
               what=f"{rows}x{cols} nvec={nvec}")
    assert tc_engine.epq_device_error() == 0


def test_tc_one_hot_is_exact_column(tc_engine, cuda_dev):
    """A one-hot x returns a column of deq(W) bit for bit: one nonzero
    product per row, exact scaling, a single rounding of n*S - M."""
    rows, cols = 96, 1024
    W = synthetic.student_t((rows, cols), seed=77).numpy()
    packed = oracle.quantize(Q4K, W)
    deq = oracle.dequantize(Q4K, packed, cols)
    js = [0, 1, 2, 3, 4, 5, 6, 7, 8, 31, 32, 63, 255, 256, 300, 777, 1023]
    pk = torch.from_numpy(packed).to(cuda_dev)
    for j in js:
        x = np.zeros((1, cols), np.float32)
        x[0, j] = 1.0
        y = tc_engine.epq_gemv(Q4K, pk, torch.from_numpy(x).to(cuda_dev), rows, cols).cpu().numpy()
        assert np.array_equal(y[0], deq[:, j]), j


def test_tc_scales_and_dynamic_range(tc_engine, cuda_dev):
    """Vectors of very different magnitudes, and a vector whose superblocks
    differ by 2^40 in magnitude (each superblock has its own operand scale)."""
    rows, cols = 300, 4096
    W = synthetic.student_t((rows, cols), seed=91).numpy()
    packed = oracle.quantize(Q4K, W)
    x = synthetic.normal((8, cols), seed=92).numpy()
    x = (x * np.float32(10.0) ** np.arange(-20, 20, 5, dtype=np.float32)[:, None]).astype(np.float32)
    x[7] = x[7] / np.float32(1e15) * np.float32(2.0) ** ((np.arange(cols) // 256) * 2.5).astype(np.float32)
    y = tc_engine.epq_gemv(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                           rows, cols).cpu().numpy()
    _check(y, oracle.gemv_f64(Q4K, packed, x, cols), oracle.gemv_bound(Q4K, packed, x, cols), what="scales")


def test_tc_zero_x_and_deterministic(tc_engine, cuda_dev):
    rows, cols = 513, 4096
    W = synthetic.student_t((rows, cols), seed=4).numpy()
    packed = oracle.quantize(Q4K, W)
    x = synthetic.normal((2, cols), seed=5).numpy()
    pk = torch.from_numpy(packed).to(cuda_dev)
    xs = torch.from_numpy(x).to(cuda_dev)
    y0 = tc_engine.epq_gemv(Q4K, pk, torch.zeros_like(xs), rows, cols)
    assert (y0 == 0).all()
    ys = [tc_engine.epq_gemv(Q4K, pk, xs, rows, cols) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


@pytest.mark.parametrize("shape", [(200, 2048), (1500, 4096), (64, 14336)])
def test_tc_residual_and_prenorm(tc_engine, cuda_dev, shape):
    rows, cols = shape
    nvec, eps = 2, 1e-6
    W = synthetic.student_t((rows, cols), seed=11).numpy()
    packed = oracle.quantize(Q4K, W)
    x = (synthetic.normal((nvec, cols), seed=12).numpy() * 3.0).astype(np.float32)
    res = synthetic.normal((nvec, rows), seed=13).numpy()
    pk = torch.from_numpy(packed).to(cuda_dev)
    y = torch.from_numpy(res).to(cuda_dev).clone()  # in-place residual update
    tc_engine.epq_gemv_ex(Q4K, pk, torch.from_numpy(x).to(cuda_dev), rows, cols, y=y, residual=y,
                          rms_prenorm=True, rms_eps=eps)
    xn = oracle.rmsnorm_f64(x, eps)
    ref = res + oracle.gemv_f64(Q4K, packed, xn, cols)
    A = oracle.gemv_bound(Q4K, packed, xn, cols) + np.abs(res)
    _check(y.cpu().numpy(), ref, A, what="residual+prenorm")


@pytest.mark.parametrize("shape", [(333, 1024), (2000, 4096), (40, 8192)])
def test_tc_swiglu(tc_engine, cuda_dev, shape):
    I, cols = shape
    nvec = 2
    W = synthetic.student_t((2 * I, cols), seed=21).numpy()
    packed = oracle.quantize(Q4K, W)
    x = synthetic.normal((nvec, cols), seed=22).numpy()
    h = tc_engine.epq_gemv_ex(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                              2 * I, cols, swiglu=True).cpu().numpy()
    y = oracle.gemv_f64(Q4K, packed, x, cols)
    A = oracle.gemv_bound(Q4K, packed, x, cols)
    g, u = y[:, :I], y[:, I:]
    Ag, Au = A[:, :I], A[:, I:]
    silu = g / (1 + np.exp(-g))
    ref = silu * u
    bound = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(ref)
    err = np.abs(h - ref)
    assert (err <= bound + 1e-30).all(), (err / (bound + 1e-30)).max()


def test_tc_grouped_heads(tc_engine, cuda_dev):
    rows, cols, hd, grp = 64, 4096, 128, 4
    W = synthetic.student_t((rows, cols), seed=31).numpy()
    packed = oracle.quantize(Q4K, W)
    v = synthetic.normal((1, cols // grp), seed=32).numpy()
    xe = np.stack([np.concatenate([np.tile(v[0, h * hd:(h + 1) * hd], grp) for h in range(cols // grp // hd)])])
    y = tc_engine.epq_gemv_ex(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(v).to(cuda_dev),
                              rows, cols, x_group=grp, x_head_dim=hd).cpu().numpy()
    _check(y, oracle.gemv_f64(Q4K, packed, xe, cols), oracle.gemv_bound(Q4K, packed, xe, cols), what="grouped")


def test_tc_full_size_sampled(tc_engine, cuda_dev):
    """Full 8B shapes (q, gate/up, down, LM head) through the engine; the
    oracle recomputes a seeded sample of 128 rows of each."""
    for rows, cols in ((4096, 4096), (28672, 4096), (4096, 14336), (128256, 4096)):
        W = synthetic.student_t((rows, cols), seed=rows + cols, device=cuda_dev)
        x = synthetic.normal((2, cols), seed=5, device=cuda_dev)
        blocks = tc_engine.epq_quantize(Q4K, W)
        y = tc_engine.epq_gemv(Q4K, blocks, x, rows, cols)
        idx = torch.randperm(rows, generator=torch.Generator().manual_seed(rows))[:128].sort().values
        # the oracle packs the sampled rows itself; the GPU's packing must match bit for bit
        packed = oracle.quantize(Q4K, W[idx.to(cuda_dev)].cpu().numpy())
        assert np.array_equal(packed, blocks[idx.to(cuda_dev)].cpu().numpy())
        xs = x.cpu().numpy()
        _check(y[:, idx.to(cuda_dev)].cpu().numpy(), oracle.gemv_f64(Q4K, packed, xs, cols),
               oracle.gemv_bound(Q4K, packed, xs, cols), what=f"full {rows}x{cols}")
        del W, blocks


@pytest.mark.parametrize("nvec", [3, 4, 5, 8])
@pytest.mark.parametrize("rows", [1, 9, 1234])
def test_tc_multi_vector_one_pass(tc_engine, cuda_dev, nvec, rows):
    """3..8 vectors over 4096-column rows share one weight pass."""
    cols = 4096
    W = synthetic.student_t((rows, cols), seed=rows + nvec).numpy()
    packed = oracle.quantize(Q4K, W)
    blocks = torch.from_numpy(packed).to(cuda_dev)
    x = synthetic.normal((nvec, cols), seed=7 + nvec).numpy()
    x = (x * np.float32(4.0) ** np.arange(nvec, dtype=np.float32)[:, None]).astype(np.float32)
    y = tc_engine.epq_gemv(Q4K, blocks, torch.from_numpy(x).to(cuda_dev), rows, cols).cpu().numpy()
    _check(y, oracle.gemv_f64(Q4K, packed, x, cols), oracle.gemv_bound(Q4K, packed, x, cols),
           what=f"{rows} rows nvec={nvec}")


@pytest.mark.parametrize("nvec", [4, 8])
def test_tc_multi_vector_options(tc_engine, cuda_dev, nvec):
    """SwiGLU pairs, residual + RMS pre-norm and grouped heads with 4 and 8 vectors."""
    cols, I, rows, eps = 4096, 700, 500, 1e-6
    # SwiGLU
    W = synthetic.student_t((2 * I, cols), seed=41).numpy()
    packed = oracle.quantize(Q4K, W)
    x = synthetic.normal((nvec, cols), seed=42).numpy()
    h = tc_engine.epq_gemv_ex(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                              2 * I, cols, swiglu=True).cpu().numpy()
    y = oracle.gemv_f64(Q4K, packed, x, cols)
    A = oracle.gemv_bound(Q4K, packed, x, cols)
    g, u, Ag, Au = y[:, :I], y[:, I:], A[:, :I], A[:, I:]
    silu = g / (1 + np.exp(-g))
    bound = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(silu * u)
    assert (np.abs(h - silu * u) <= bound + 1e-30).all()
    # residual (in place) + RMS pre-norm
    W = synthetic.student_t((rows, cols), seed=43).numpy()
    packed = oracle.quantize(Q4K, W)
    res = synthetic.normal((nvec, rows), seed=44).numpy()
    yt = torch.from_numpy(res).to(cuda_dev).clone()
    tc_engine.epq_gemv_ex(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev), rows, cols,
                          y=yt, residual=yt, rms_prenorm=True, rms_eps=eps)
    xn = oracle.rmsnorm_f64(x, eps)
    _check(yt.cpu().numpy(), res + oracle.gemv_f64(Q4K, packed, xn, cols),
           oracle.gemv_bound(Q4K, packed, xn, cols) + np.abs(res), what="residual+prenorm")
    # grouped heads
    hd, grp = 128, 4
    v = synthetic.normal((nvec, cols // grp), seed=45).numpy()
    xe = np.concatenate([np.tile(v[:, k * hd:(k + 1) * hd], (1, grp)) for k in range(cols // grp // hd)], axis=1)
    yg = tc_engine.epq_gemv_ex(Q4K, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(v).to(cuda_dev), rows,
                               cols, x_group=grp, x_head_dim=hd).cpu().numpy()
    _check(yg, oracle.gemv_f64(Q4K, packed, xe, cols), oracle.gemv_bound(Q4K, packed, xe, cols), what="grouped")
