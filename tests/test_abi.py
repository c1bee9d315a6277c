"""CPU checks of the C ABI: the library builds, loads and exports every
function that include/epq.h declares; host-only queries agree with the
oracle's definitions.  No compute call is made (no GPU here)."""
import oracle


def test_exports_every_declared_symbol(epq_lib):
    lib = epq_lib.load()
    names = epq_lib.declared_symbols()
    assert "epq_gemv" in names and "epq_quantize" in names
    for n in names:
        assert hasattr(lib, n), n


def test_row_bytes_agree_with_oracle(epq_lib):
    for fmt in oracle.FORMATS:
        assert epq_lib.epq_block_weights(fmt) == oracle.BLOCK_WEIGHTS[fmt]
        assert epq_lib.epq_block_bytes(fmt) == oracle.BLOCK_BYTES[fmt]
        for cols in (0, 32, 48, 256, 512, 1000, 4096, 14336):
            assert epq_lib.epq_row_bytes(fmt, cols) == oracle.row_bytes(fmt, cols), (fmt, cols)
    assert epq_lib.epq_row_bytes(9, 256) == -1


def test_status_strings(epq_lib):
    assert epq_lib.epq_status_string(0) == "ok"
    assert "align" in epq_lib.epq_status_string(4)
    assert epq_lib.epq_status_string(99) == "unknown status"
