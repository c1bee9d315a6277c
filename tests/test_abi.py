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


def test_tuning_keys(epq_lib):
    """epq_set_tuning returns the previous value, and leaves the setting
    unchanged (returning -1) for an unknown key or a value out of range."""
    e = epq_lib
    cases = [(e.EPQ_TUNE_GEMV_ENGINE, 4, (-1, 5)), (e.EPQ_TUNE_VN_CHUNK, 5, (-1, 65)), (e.EPQ_TUNE_VN_CLUSTER, 4, (-1, 3, 8)), (e.EPQ_TUNE_TILE_BYTES, 65536, (4095, 131073)),
             (e.EPQ_TUNE_RING_BYTES, 65536, (32767, 200705)), (e.EPQ_TUNE_EARLY_STAGES, 3, (-1, 17)),
             (e.EPQ_TUNE_TC_SPLIT, 8, (3, 32)), (e.EPQ_TUNE_ATTN_CHUNK, 64, (-8, 4, 12, 4104))]
    for key, value, bad in cases:
        prev = e.epq_set_tuning(key, value)
        assert prev >= 0
        for b in bad:
            assert e.epq_set_tuning(key, b) == -1
        assert e.epq_set_tuning(key, prev) == value  # restored; the bad values changed nothing
    assert e.epq_set_tuning(99, 1) == -1


def test_chain_workspace_size(epq_lib):
    assert epq_lib.epq_gemv_chain_workspace_bytes() >= 8
