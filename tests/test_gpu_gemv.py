"""GPU parity of the dequant-GEMV against the float64 oracle.

Bar (the accuracy target of the GEMV): |y_gpu - y_ref| <= 1e-4 * sum_j |deq(W)_ij x_j|
per row and vector.  Special inputs make exact results exact: a one-hot x
returns a column of deq(W) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _case(fmt, rows, cols, nvec, seed):
    W = synthetic.student_t((rows, cols), seed=seed).numpy()
    x = synthetic.normal((nvec, cols), seed=seed + 1).numpy()
    return W, oracle.quantize(fmt, W), x


def _check(y_gpu, y_ref, A, tol=TOL, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    lim = tol * A + 1e-30
    bad = np.argwhere(err > lim)
    assert bad.size == 0, f"{what}: {bad.shape[0]} outputs beyond bound, first {bad[:3].tolist()}, " \
                          f"worst ratio {(err / lim).max():.3g}"


SHAPES = [(1, 256), (7, 512), (33, 1024), (130, 4096), (257, 2048), (20, 14336), (1000, 768), (3, 1280)]


@pytest.mark.parametrize("fmt", oracle.FORMATS)
@pytest.mark.parametrize("shape", SHAPES)
def test_gemv_parity(epq_lib, cuda_dev, fmt, shape):
    rows, cols = shape
    for nvec in (1, 2, 3):
        W, packed, x = _case(fmt, rows, cols, nvec, seed=rows * 31 + cols + fmt * 7 + nvec)
        y = epq_lib.epq_gemv(fmt, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                             rows, cols).cpu().numpy()
        _check(y, oracle.gemv_f64(fmt, packed, x, cols), oracle.gemv_bound(fmt, packed, x, cols),
               what=f"fmt={fmt} {rows}x{cols} nvec={nvec}")
    assert epq_lib.epq_device_error() == 0


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_nvec8_and_scales(epq_lib, cuda_dev, fmt):
    """Eight verify vectors with very different magnitudes (1e-20 .. 1e20)."""
    rows, cols = 300, 4096
    W, packed, x = _case(fmt, rows, cols, 8, seed=500 + fmt)
    x = x * np.float32(10.0) ** np.arange(-20, 20, 5, dtype=np.float32)[:, None]
    x = x.astype(np.float32)
    y = epq_lib.epq_gemv(fmt, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                         rows, cols).cpu().numpy()
    _check(y, oracle.gemv_f64(fmt, packed, x, cols), oracle.gemv_bound(fmt, packed, x, cols), what="nvec8")


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_one_hot_is_exact_column(epq_lib, cuda_dev, fmt):
    rows, cols = 96, 512
    W, packed, _ = _case(fmt, rows, cols, 1, seed=900 + fmt)
    deq = oracle.dequantize(fmt, packed, cols)
    js = [0, 1, 5, 6, 7, 8, 31, 32, 255, 256, 300, 511]
    x = np.zeros((len(js), cols), np.float32)
    for v, j in enumerate(js):
        x[v, j] = 1.0
    pk = torch.from_numpy(packed).to(cuda_dev)
    y = np.concatenate([epq_lib.epq_gemv(fmt, pk, torch.from_numpy(x[v0:v0 + 6]).to(cuda_dev), rows, cols)
                        .cpu().numpy() for v0 in range(0, len(js), 6)])
    for v, j in enumerate(js):
        assert np.array_equal(y[v], deq[:, j]), (fmt, j)


def test_gemv_zero_x_and_deterministic(epq_lib, cuda_dev):
    fmt, rows, cols = oracle.Q4_K, 513, 4096
    W, packed, x = _case(fmt, rows, cols, 2, seed=4)
    pk = torch.from_numpy(packed).to(cuda_dev)
    xs = torch.from_numpy(x).to(cuda_dev)
    y0 = epq_lib.epq_gemv(fmt, pk, torch.zeros_like(xs), rows, cols)
    assert (y0 == 0).all()
    ys = [epq_lib.epq_gemv(fmt, pk, xs, rows, cols) for _ in range(3)]
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q4_0, oracle.Q2_K, oracle.Q6_K])
def test_gemv_ex_residual_and_prenorm(epq_lib, cuda_dev, fmt):
    rows, cols, nvec, eps = 200, 2048, 2, 1e-6
    W, packed, x = _case(fmt, rows, cols, nvec, seed=11)
    x = (x * 3.0).astype(np.float32)
    res = synthetic.normal((nvec, rows), seed=12).numpy()
    pk = torch.from_numpy(packed).to(cuda_dev)
    y = torch.from_numpy(res).to(cuda_dev).clone()          # in-place residual update
    epq_lib.epq_gemv_ex(fmt, pk, torch.from_numpy(x).to(cuda_dev), rows, cols, y=y, residual=y,
                        rms_prenorm=True, rms_eps=eps)
    xn = oracle.rmsnorm_f64(x, eps)
    ref = res + oracle.gemv_f64(fmt, packed, xn, cols)
    A = oracle.gemv_bound(fmt, packed, xn, cols) + np.abs(res)
    _check(y.cpu().numpy(), ref, A, what="residual+prenorm")


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_ex_swiglu(epq_lib, cuda_dev, fmt):
    I, cols, nvec = 333, 1024, 2
    W, packed, x = _case(fmt, 2 * I, cols, nvec, seed=21 + fmt)
    h = epq_lib.epq_gemv_ex(fmt, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(x).to(cuda_dev),
                            2 * I, cols, swiglu=True).cpu().numpy()
    y = oracle.gemv_f64(fmt, packed, x, cols)
    A = oracle.gemv_bound(fmt, packed, x, cols)
    g, u = y[:, :I], y[:, I:]
    Ag, Au = A[:, :I], A[:, I:]
    sig = 1 / (1 + np.exp(-g))
    silu = g * sig
    ref = silu * u
    # |d silu/dg| <= 1.1; errors of g and u propagate through the product
    bound = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(ref)
    err = np.abs(h - ref)
    assert (err <= bound + 1e-30).all(), (err / (bound + 1e-30)).max()


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q2_K, oracle.Q6_K])
def test_gemv_ex_grouped_heads(epq_lib, cuda_dev, fmt):
    """x_group: each 128-float head of x feeds 4 consecutive heads of the product."""
    rows, cols, hd, grp = 64, 4096, 128, 4
    W, packed, _ = _case(fmt, rows, cols, 1, seed=31)
    v = synthetic.normal((1, cols // grp), seed=32).numpy()
    xe = np.stack([np.concatenate([np.tile(v[0, h * hd:(h + 1) * hd], grp) for h in range(cols // grp // hd)])])
    y = epq_lib.epq_gemv_ex(fmt, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(v).to(cuda_dev),
                            rows, cols, x_group=grp, x_head_dim=hd).cpu().numpy()
    _check(y, oracle.gemv_f64(fmt, packed, xe, cols), oracle.gemv_bound(fmt, packed, xe, cols), what="grouped")


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_gemv_full_size_layer_sampled(epq_lib, cuda_dev, fmt):
    """Full 8B-layer shapes in the launch configuration the bench uses; the
    oracle recomputes a seeded sample of 128 rows of each matrix."""
    for rows, cols in ((4096, 4096), (14336, 4096), (4096, 14336), (1024, 4096)):
        W = synthetic.student_t((rows, cols), seed=rows + cols + fmt, device=cuda_dev)
        x = synthetic.normal((1, cols), seed=5, device=cuda_dev)
        blocks = epq_lib.epq_quantize(fmt, W)
        y = epq_lib.epq_gemv(fmt, blocks, x, rows, cols)
        idx = torch.randperm(rows, generator=torch.Generator().manual_seed(rows + fmt))[:128].sort().values
        Ws = W[idx.to(cuda_dev)].cpu().numpy()
        packed = oracle.quantize(fmt, Ws)
        assert np.array_equal(packed, blocks[idx.to(cuda_dev)].cpu().numpy())
        xs = x.cpu().numpy()
        _check(y[:, idx.to(cuda_dev)].cpu().numpy(), oracle.gemv_f64(fmt, packed, xs, cols),
               oracle.gemv_bound(fmt, packed, xs, cols), what=f"full {rows}x{cols}")


def test_gemv_argument_errors(epq_lib, cuda_dev):
    pk = torch.zeros((4, 144), dtype=torch.uint8, device=cuda_dev)
    x = torch.zeros((1, 256), device=cuda_dev)
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv(3, pk, torch.zeros((9, 256), device=cuda_dev), 4, 256)   # nvec > 8
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv(3, pk, x, 4, 128)                                       # cols % 256
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv(3, pk, x, 0, 256)                                       # rows < 1
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_gemv(3, pk, x, 4, 32768)                                     # cols too large


@pytest.fixture
def engine3(epq_lib):
    """The block-diagonal tensor-core engine for the Q4_K GEMVs."""
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, 3)
    yield
    epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


@pytest.mark.parametrize("shape", SHAPES)
def test_q4k_block_diagonal_engine_parity(epq_lib, cuda_dev, engine3, shape):
    test_gemv_parity(epq_lib, cuda_dev, oracle.Q4_K, shape)


def test_q4k_block_diagonal_engine_options(epq_lib, cuda_dev, engine3):
    test_gemv_nvec8_and_scales(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_one_hot_is_exact_column(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_ex_residual_and_prenorm(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_ex_swiglu(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_ex_grouped_heads(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_full_size_layer_sampled(epq_lib, cuda_dev, oracle.Q4_K)


@pytest.fixture
def engine4(epq_lib):
    """The vector-column tensor-core engine for the Q4_K GEMVs of 2+ vectors."""
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, 4)
    yield
    epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_GEMV_ENGINE, prev)


MULTI_SHAPES = [(130, 4096, 4), (257, 2048, 5), (300, 4096, 8), (20, 14336, 6), (1000, 768, 7), (64, 256, 3),
                (48, 1024, 2)]


@pytest.mark.parametrize("rows,cols,nvec", MULTI_SHAPES)
def test_q4k_block_diagonal_vectors_in_one_pass(epq_lib, cuda_dev, engine3, rows, cols, nvec):
    """Up to 8 vectors per weight pass (4 or 8 x-operand sets in shared
    memory; rows of 14336 take passes of two)."""
    _multi_vector_case(epq_lib, cuda_dev, rows, cols, nvec)


@pytest.mark.parametrize("cluster", [0, 1, 4])
@pytest.mark.parametrize("chunk", [0, 3, 7])
@pytest.mark.parametrize("rows,cols,nvec", MULTI_SHAPES)
def test_q4k_vector_column_engine(epq_lib, cuda_dev, engine4, rows, cols, nvec, chunk, cluster):
    """The vector-column engine (8 vector columns per MMA): the whole row's x
    operands in shared memory, or chunks of 3 / 7 superblocks with partial
    sums kept between chunks (rows of 14336 are chunked by default); the x
    conversion shared by clusters of 2 (automatic) or 4 CTAs, or not."""
    prev = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_VN_CHUNK, chunk)
    prev_cl = epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_VN_CLUSTER, cluster)
    try:
        _multi_vector_case(epq_lib, cuda_dev, rows, cols, nvec)
    finally:
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_VN_CHUNK, prev)
        epq_lib.epq_set_tuning(epq_lib.EPQ_TUNE_VN_CLUSTER, prev_cl)


def test_q4k_vector_column_engine_options(epq_lib, cuda_dev, engine4):
    test_gemv_nvec8_and_scales(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_one_hot_is_exact_column(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_ex_residual_and_prenorm(epq_lib, cuda_dev, oracle.Q4_K)
    test_gemv_ex_swiglu(epq_lib, cuda_dev, oracle.Q4_K)
    for shape in SHAPES:
        test_gemv_parity(epq_lib, cuda_dev, oracle.Q4_K, shape)


def test_q4k_vector_column_engine_grouped_heads(epq_lib, cuda_dev, engine4):
    """x_group with 4 vectors: each 128-float head of a vector feeds 4
    consecutive heads of the product."""
    fmt, rows, cols, hd, grp, nvec = oracle.Q4_K, 64, 4096, 128, 4, 4
    W, packed, _ = _case(fmt, rows, cols, 1, seed=41)
    v = synthetic.normal((nvec, cols // grp), seed=42).numpy()
    xe = np.stack([np.concatenate([np.tile(v[k, h * hd:(h + 1) * hd], grp) for h in range(cols // grp // hd)])
                   for k in range(nvec)])
    y = epq_lib.epq_gemv_ex(fmt, torch.from_numpy(packed).to(cuda_dev), torch.from_numpy(v).to(cuda_dev),
                            rows, cols, x_group=grp, x_head_dim=hd).cpu().numpy()
    _check(y, oracle.gemv_f64(fmt, packed, xe, cols), oracle.gemv_bound(fmt, packed, xe, cols), what="grouped")


def test_q4k_vector_column_engine_full_size_sampled(epq_lib, cuda_dev, engine4):
    """8 vectors on the full 8B-layer shapes (the down projection chunked)."""
    fmt = oracle.Q4_K
    for rows, cols in ((14336, 4096), (4096, 14336)):
        W = synthetic.student_t((rows, cols), seed=rows + 3 * cols, device=cuda_dev)
        pk = epq_lib.epq_quantize(fmt, W)
        x = synthetic.normal((8, cols), seed=cols + 9).to(cuda_dev)
        y = epq_lib.epq_gemv(fmt, pk, x, rows, cols).cpu().numpy()
        idx = np.sort(np.random.default_rng(rows).choice(rows, 128, replace=False))
        pks = oracle.quantize(fmt, W.cpu().numpy()[idx])   # the oracle packs its own rows ...
        assert np.array_equal(pks, pk.cpu().numpy()[idx])   # ... which the GPU packer matches byte for byte
        xs = x.cpu().numpy()
        _check(y[:, idx], oracle.gemv_f64(fmt, pks, xs, cols), oracle.gemv_bound(fmt, pks, xs, cols), what="full")
    assert epq_lib.epq_device_error() == 0


def _multi_vector_case(epq_lib, cuda_dev, rows, cols, nvec):
    """Plain, SwiGLU and residual + RMS pre-norm with nvec vectors, each
    vector with its own magnitude so that a vector reading another's
    operands or RMS factor fails."""
    fmt, eps = oracle.Q4_K, 1e-6
    W, packed, x = _case(fmt, rows, cols, nvec, seed=rows * 7 + cols + nvec)
    x = (x * np.float32(10.0) ** np.arange(-3, nvec - 3, dtype=np.float32)[:, None]).astype(np.float32)
    pk = torch.from_numpy(packed).to(cuda_dev)
    xd = torch.from_numpy(x).to(cuda_dev)
    y = epq_lib.epq_gemv(fmt, pk, xd, rows, cols).cpu().numpy()
    _check(y, oracle.gemv_f64(fmt, packed, x, cols), oracle.gemv_bound(fmt, packed, x, cols), what="plain")
    res = synthetic.normal((nvec, rows), seed=rows + 5).numpy()
    yr = torch.from_numpy(res).to(cuda_dev).clone()
    epq_lib.epq_gemv_ex(fmt, pk, xd, rows, cols, y=yr, residual=yr, rms_prenorm=True, rms_eps=eps)
    xn = oracle.rmsnorm_f64(x, eps)
    _check(yr.cpu().numpy(), res + oracle.gemv_f64(fmt, packed, xn, cols),
           oracle.gemv_bound(fmt, packed, xn, cols) + np.abs(res), what="residual+prenorm")
    I = rows // 2
    h = epq_lib.epq_gemv_ex(fmt, pk[:2 * I], xd, 2 * I, cols, swiglu=True).cpu().numpy()
    yy = oracle.gemv_f64(fmt, packed[:2 * I], x, cols)
    A = oracle.gemv_bound(fmt, packed[:2 * I], x, cols)
    g, u, Ag, Au = yy[:, :I], yy[:, I:], A[:, :I], A[:, I:]
    silu = g / (1 + np.exp(-g))
    ref = silu * u
    bound = TOL * (1.1 * Ag * np.abs(u) + np.abs(silu) * Au) + 1e-6 * np.abs(ref)
    assert (np.abs(h - ref) <= bound + 1e-30).all(), (np.abs(h - ref) / (bound + 1e-30)).max()
    assert epq_lib.epq_device_error() == 0
