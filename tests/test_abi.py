"""The C-ABI library loads and exports every entry point its header declares.
Only host-side calls are made here (no GPU in this environment)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spc_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def spc():
    import bit_kv_cache_spc_gb300 as m
    return m


def test_header_declares_the_hot_path():
    names = declared_functions()
    for fn in ("spc_quantize_kv", "spc_decode_attn2", "spc_topk_select", "spc_host_gather", "spc_merged_attn",
               "spc_merged_attn_fetch", "spc_append_kv", "spc_topk_select_prev", "spc_merged_attn_fetch_prev"):
        assert fn in names


def test_every_declared_symbol_is_exported(spc):
    lib = C.CDLL(spc.lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_queries(spc):
    assert spc.spc_abi_version() == 2
    d = spc.Dims(1, 32, 8, 32768, 128, 1)
    assert spc.spc_num_quantized(d) == 32640
    assert spc.spc_records_bytes(d) == 8 * 1020 * 2048
    assert spc.spc_resid_bytes(d) == 8 * 128 * 2 * 128 * 2
    d2 = spc.Dims(16, 32, 32, 2048, 128, 2)
    assert spc.spc_records_bytes(d2) == 16 * 32 * 60 * 3072  # 96 B per token and KV head
    bad = spc.Dims(1, 32, 8, 1024, 32, 3)
    assert spc.spc_num_quantized(bad) == -1


def test_validation_happens_before_any_launch(spc):
    """Argument errors come back as status codes; nothing reaches the GPU."""
    bad_bits = spc.Dims(1, 32, 8, 1024, 32, 3)
    with pytest.raises(spc.SpcError) as e:
        spc.spc_quantize_kv(bad_bits, 16, 16, 16, 16, stream=0)
    assert e.value.status == 1
    g8 = spc.Dims(1, 64, 8, 1024, 32, 1)
    with pytest.raises(spc.SpcError) as e:
        spc.spc_topk_select(g8, 16, 16, 4, 16, 16, stream=0)
    assert e.value.status == 2
    d = spc.Dims(1, 32, 8, 1024, 32, 1)
    with pytest.raises(spc.SpcError) as e:  # misaligned query pointer
        spc.spc_decode_attn2(d, 16, 16, 18, 16, None, None, 16, 1 << 30, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # misaligned self row of the speculative token
        spc.spc_merged_attn(d, 16, 16, 16, None, None, None, 0, 16, None, None, 16, 1 << 30, stream=0, kv_self=20)
    assert e.value.status == 1
    small_cap = spc.Dims(1, 32, 8, 1024, 32, 1, q_groups_cap=3)
    with pytest.raises(spc.SpcError) as e:
        spc.spc_quantize_kv(small_cap, 16, 16, 16, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # negative k
        spc.spc_topk_select(d, 16, 16, -1, 16, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # speculative logits not on a 16-byte boundary
        spc.spc_topk_select(d, 20, 16, 4, 16, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the selection with its previous slots: no src output
        spc.spc_topk_select_prev(d, 16, 16, 4, 16, 16, 32, 4, None, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the previous selection is the output
        spc.spc_topk_select_prev(d, 16, 16, 4, 16, 16, 16, 4, 48, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # ... or overlaps it (8 KV heads x 4 entries x 4 B = 128 B per buffer)
        spc.spc_topk_select_prev(d, 16, 16, 4, 1024, 16, 1024 + 64, 4, 48, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # a pre-fetch that keeps staged rows needs src
        spc.spc_merged_attn_fetch_prev(d, 16, 16, 16, None, None, None, 0, 16, None, None, 16, 64, 1024, 16, 4, 32,
                                       None, 48, 4, ws_bytes=1 << 30, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the fused step with kept rows: no next_src
        spc.spc_decode_step_prev(d, 16, 16, 16, 16, 16, 16, 4, 16, 16, 16, 4, 32, 48, None, 64, ws_bytes=1 << 30,
                                 stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # ... or next_idx the same buffer as idx
        spc.spc_decode_step_prev(d, 16, 16, 16, 16, 16, 16, 4, 16, 16, 16, 4, 16, 48, 80, 64, ws_bytes=1 << 30,
                                 stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the standalone pre-fetch with kept rows needs src too
        spc.spc_host_gather_prev(d, 64, 1024, 16, 4, 32, None, 48, 4, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # ... and a previous staging other than its output
        spc.spc_host_gather_prev(d, 64, 1024, 16, 4, 32, 80, 32, 4, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # ... and a previous staging other than its output
        spc.spc_merged_attn_fetch_prev(d, 16, 16, 16, None, None, None, 0, 16, None, None, 16, 64, 1024, 16, 4, 32,
                                       64, 32, 4, ws_bytes=1 << 30, stream=0)
    assert e.value.status == 1
    # staging buffers that share bytes: one row of this shape's staging is 8 KV heads x 512 B = 4096 B per k
    row = 8 * 512
    with pytest.raises(spc.SpcError) as e:  # the carried copy would write rows the attention reads
        spc.spc_merged_attn_fetch(d, 16, 16, 16, 32, 48, 1 << 20, 4, 16, None, None, 16, 64, 1024, 16, 4,
                                  (1 << 20) + 3 * row, ws_bytes=1 << 30, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # ... also with kept rows: the previous staging overlaps the output
        spc.spc_merged_attn_fetch_prev(d, 16, 16, 16, 32, 48, 1 << 20, 4, 16, None, None, 16, 64, 1024, 16, 4,
                                       1 << 24, 32, (1 << 24) - 2 * row, 4, ws_bytes=1 << 30, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the fused step: its carried copy over the rows it reads
        spc.spc_decode_step(d, 16, 16, 16, 32, 48, 1 << 20, 4, 16, 16, 16, 4, 64, 80, 96, ws_bytes=1 << 30,
                            fetch_host_kv=64, fetch_n_cap=1024, fetch_idx=16, fetch_k=4,
                            fetch_staging=(1 << 20) + row, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # the standalone gather with kept rows, overlapping by one byte range
        spc.spc_host_gather_prev(d, 64, 1024, 16, 4, 1 << 20, 32, (1 << 20) + row, 4, stream=0)
    assert e.value.status == 1


def test_kernel_count_queries_refuse_bad_arguments(spc):
    """The launch-count queries answer -1 for an invalid shape or count (no
    launch; their positive answers depend on the device and are checked on
    the GPU)."""
    bad_bits = spc.Dims(1, 32, 8, 1024, 32, 3)
    assert spc.spc_attn_kernel_count(bad_bits, 0, 0) == -1
    assert spc.spc_decode_step_kernel_count(bad_bits, 8, 0, 8) == -1
    d = spc.Dims(1, 32, 8, 1024, 32, 1)
    assert spc.spc_attn_kernel_count(d, -1, 0) == -1
    assert spc.spc_attn_kernel_count(d, 0, -1) == -1
    assert spc.spc_decode_step_kernel_count(d, 8, 0, -1) == -1


def test_append_validation(spc):
    """The append needs room for the new window row and, at a flush, for the
    new record; both are checked before any launch."""
    d = spc.Dims(1, 32, 8, 1000, 32, 1)  # resid_cap defaults to exactly r: no room
    with pytest.raises(spc.SpcError) as e:
        spc.spc_append_kv(d, 16, 16, 16, 16, stream=0)
    assert e.value.status == 1
    # N = 1023, R = 32: the 1024th token completes group 30 (N_q 960 -> 992)
    full = spc.Dims(1, 32, 8, 1023, 32, 1, resid_cap=64)
    assert spc.spc_num_quantized(full) == 960
    with pytest.raises(spc.SpcError) as e:  # q_groups_cap = 30 has no slot for record 30
        spc.spc_append_kv(full, 16, 16, 16, 16, stream=0)
    assert e.value.status == 1
    ok_caps = spc.Dims(1, 32, 8, 1023, 32, 1, q_groups_cap=31, resid_cap=64)
    with pytest.raises(spc.SpcError) as e:  # misaligned new key row
        spc.spc_append_kv(ok_caps, 18, 16, 16, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(spc.SpcError) as e:  # host cache too short for row N
        spc.spc_append_kv(ok_caps, 16, 16, 16, 16, host_kv=16, n_cap=1023, stream=0)
    assert e.value.status == 1


def test_group_size_validation(spc):
    """g = 32 and 64 are accepted (N_q is a whole number of groups); other sizes are refused."""
    assert spc.spc_num_quantized(spc.Dims(1, 32, 8, 1000, 40, 1, group=64)) == 960
    assert spc.spc_num_quantized(spc.Dims(1, 32, 8, 1000, 40, 1)) == 960
    assert spc.spc_num_quantized(spc.Dims(1, 32, 8, 1100, 40, 1, group=64)) == 1024
    d48 = spc.Dims(1, 32, 8, 1000, 40, 1)
    d48.group = 48
    with pytest.raises(spc.SpcError) as e:
        spc.spc_quantize_kv(d48, 16, 16, 16, 16, stream=0)
    assert e.value.status == 2


def test_pipeline_refuses_a_schedule_that_reads_its_own_fetch(spc):
    """DecodePipeline checks the layer count and the lag before it touches a
    device: at lag = L a layer's attention would carry the fetch of the rows it
    reads, and lag 0 is the same layer."""
    from bit_kv_cache_spc_gb300.pipeline import DecodePipeline
    d = spc.Dims(1, 4, 1, 1024, 64, 1)
    for n_layers, lag in ((2, 2), (3, 3), (3, 0), (1, 1), (4, 7)):
        rec = [object()] * n_layers
        with pytest.raises(ValueError):
            DecodePipeline(d, 24, rec, rec, rec, 1024, rec, rec, rec, rec, None, 0, lag=lag)
