"""GPU parity of the packer and unpacker: bit-exact with the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

SHAPES = [(1, 256), (3, 512), (37, 4096), (5, 14336), (130, 1024)]


def _special_rows(cols):
    """Degenerate and boundary rows: zeros, -0, constants, all-positive,
    all-negative, ties at the largest magnitude, tiny values (fp16
    subnormal factors), values that round at exact .5 code boundaries."""
    rows = []
    rows.append(np.zeros(cols, np.float32))
    rows.append(-np.zeros(cols, np.float32))
    rows.append(np.full(cols, 0.3, np.float32))
    rows.append(np.full(cols, -0.7, np.float32))
    r = np.abs(np.linspace(0.01, 1.0, cols, dtype=np.float32))
    rows.append(r)
    rows.append(-r)
    t = np.array([((j % 16) - 8) / 4 for j in range(cols)], np.float32)
    t[5::32] = 2.0                           # +2 and -2 tie for the largest magnitude
    rows.append(t)
    rows.append((np.arange(cols, dtype=np.float32) % 7 - 3) * np.float32(1e-6))   # subnormal fp16 factors
    rows.append((np.arange(cols, dtype=np.float32) % 32) * np.float32(0.5))        # .5 ties in the codes
    rows.append(np.where(np.arange(cols) % 32 == 0, 60000.0, 1.0).astype(np.float32))
    return np.stack(rows)


def _weights(rows, cols, seed):
    return synthetic.student_t((rows, cols), seed=seed).numpy()


@pytest.mark.parametrize("fmt", oracle.FORMATS)
@pytest.mark.parametrize("shape", SHAPES)
def test_quantize_bitexact(epq_lib, cuda_dev, fmt, shape):
    rows, cols = shape
    W = _weights(rows, cols, seed=1000 + rows * 7 + cols + fmt)
    blocks = epq_lib.epq_quantize(fmt, torch.from_numpy(W).to(cuda_dev))
    torch.cuda.synchronize()
    ref = oracle.quantize(fmt, W)
    got = blocks.cpu().numpy()
    assert got.shape == ref.shape
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"first mismatches at {bad[:5].tolist()}"
    assert epq_lib.epq_device_error() == 0


@pytest.mark.parametrize("fmt", oracle.FORMATS)
def test_quantize_special_rows(epq_lib, cuda_dev, fmt):
    for cols in (256, 512):
        W = _special_rows(cols)
        blocks = epq_lib.epq_quantize(fmt, torch.from_numpy(W).to(cuda_dev))
        ref = oracle.quantize(fmt, W)
        got = blocks.cpu().numpy()
        for r in range(W.shape[0]):
            assert got[r].tobytes() == ref[r].tobytes(), (cols, r)


@pytest.mark.parametrize("fmt", oracle.FORMATS)
@pytest.mark.parametrize("shape", [(1, 256), (37, 4096), (5, 14336)])
def test_dequantize_bitexact(epq_lib, cuda_dev, fmt, shape):
    rows, cols = shape
    W = np.concatenate([_weights(rows, cols, seed=77 + fmt), _special_rows(cols)])
    packed = oracle.quantize(fmt, W)
    out = epq_lib.epq_dequantize(fmt, torch.from_numpy(packed).to(cuda_dev), W.shape[0], cols)
    ref = oracle.dequantize(fmt, packed, cols)
    got = out.cpu().numpy()
    # compare bit patterns (distinguishes -0 from +0)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_quantize_full_size_sampled(epq_lib, cuda_dev):
    """Full 8B-layer gate matrix (14336 x 4096) packed on the GPU; a seeded
    sample of 256 rows is compared byte for byte with the oracle."""
    rows, cols = 14336, 4096
    W = synthetic.student_t((rows, cols), seed=4242, device=cuda_dev)
    for fmt in oracle.FORMATS:
        blocks = epq_lib.epq_quantize(fmt, W)
        idx = torch.randperm(rows, generator=torch.Generator().manual_seed(fmt))[:256].sort().values
        ref = oracle.quantize(fmt, W[idx.to(cuda_dev)].cpu().numpy())
        got = blocks[idx.to(cuda_dev)].cpu().numpy()
        assert np.array_equal(got, ref), oracle.formats.NAMES[fmt]


def test_argument_errors(epq_lib, cuda_dev):
    W = torch.zeros((4, 256), device=cuda_dev)
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_quantize(9, W)                       # unknown format
    with pytest.raises(epq_lib.EpqError):
        epq_lib.epq_quantize(3, torch.zeros((4, 128), device=cuda_dev))   # cols % 256
    Wbig = torch.zeros(4 * 256 + 1, device=cuda_dev)
    with pytest.raises(epq_lib.EpqError) as e:
        epq_lib.epq_quantize(3, Wbig[1:].view(4, 256))  # misaligned
    assert e.value.status == 4
