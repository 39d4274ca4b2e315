"""The C-ABI library builds, loads and exports every entry point include/msa.h
declares; host-side argument checks return statuses without touching a GPU."""
import ctypes
import os
import re

import pytest

from block_sparse_paged_msa_gb300 import build as msa_build
from block_sparse_paged_msa_gb300 import ops
from block_sparse_paged_msa_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "msa.h")


@pytest.fixture(scope="module")
def lib():
    msa_build.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps every one of them
    assert set(names) <= set(ops._SIGNATURES), set(names) - set(ops._SIGNATURES)


def test_block_counts_from_tokens(lib):
    """The library resolves sglang's token counts into block counts
    (MiniMaxSparseAttnBackend.__init__); values at the golden file's cases."""
    import json
    gold = json.load(open(os.path.join(os.path.dirname(HEADER), "..", "tests", "golden",
                                       "config_resolution.json")))
    P = gold["block_size"]
    for tokens, blocks in gold["local"]:
        assert lib.msa_local_blocks_from_tokens(tokens, P) == blocks, tokens
        assert ops.local_blocks_from_tokens(tokens, P) == blocks, tokens
    for tokens, blocks in gold["init"]:
        assert lib.msa_init_blocks_from_tokens(tokens, P) == blocks, tokens
        assert ops.init_blocks_from_tokens(tokens, P) == blocks, tokens
    assert lib.msa_local_blocks_from_tokens(-1, P) == -1
    assert lib.msa_init_blocks_from_tokens(5, 0) == -1
    with pytest.raises(ValueError):
        ops.local_blocks_from_tokens(-1, P)
    # config_for takes the library's resolution
    spec = wl.WORKLOADS["long_decode"]
    assert ops.config_for(spec).local_blocks == 5


def test_status_strings(lib):
    for s, name in ops.STATUS.items():
        assert ops.status_string(s).startswith(name)


def _cfg(**kw):
    spec = wl.small("medium_decode")
    return ops.config_for(spec, **kw)


def test_validate_config(lib):
    assert ops.validate_config(_cfg()) == 0
    assert ops.validate_config(_cfg(head_dim=64)) == 2          # unsupported
    assert ops.validate_config(_cfg(block_size=64)) == 2
    assert ops.validate_config(_cfg(index_dim=96)) == 2
    assert ops.validate_config(_cfg(num_q_heads=63)) == 1       # not a multiple
    assert ops.validate_config(_cfg(num_q_heads=8 * 17)) == 2   # group > 16
    assert ops.validate_config(_cfg(local_blocks=0)) == 1
    assert ops.validate_config(_cfg(q_len=0)) == 1
    assert ops.validate_config(_cfg(kv_dtype="fp8_e4m3", k_scale=0.0)) == 1
    assert ops.validate_config(_cfg(kv_dtype="nvfp4", k_scale=0.5, v_scale=0.5)) == 0
    assert ops.validate_config(_cfg(kv_dtype="nvfp4", v_scale=0.0)) == 1
    bad = _cfg()
    bad.kv_dtype = 3
    assert ops.validate_config(bad) == 1
    assert ops.validate_config(_cfg(softmax_scale=-1.0)) == 1


def test_workspace_and_widths(lib):
    c = _cfg()
    assert ops.selected_width(c) == 1 + 3 + 16
    n = ops.workspace_bytes(c)
    assert n > 0 and n % 256 == 0
    ns = ops.num_splits(c)
    assert 1 <= ns <= 20
    # partials dominate: T * H_q * splits * (D + 1) floats
    assert n >= 4 * c.max_batch * c.num_q_heads * ns * 129
    assert lib.msa_workspace_bytes(ctypes.byref(_cfg(head_dim=64))) == 0
    for bps, want in ((1, 20), (4, 5), (20, 1), (64, 1)):
        assert ops.num_splits(_cfg(blocks_per_split=bps)) == want


def test_host_side_errors_need_no_gpu(lib):
    c = _cfg()
    P = ctypes.c_void_p
    # null workspace / misaligned workspace / batch above max: rejected before any launch
    assert lib.msa_plan(ctypes.byref(c), 1, P(16), None, P(16), 64, None, None) == 1
    assert lib.msa_plan(ctypes.byref(c), 1, P(16), None, P(16), 64, P(258), None) == 1
    assert lib.msa_plan(ctypes.byref(c), c.max_batch + 1, P(16), None, P(16), 64, P(256),
                        None) == 1
    assert lib.msa_plan(ctypes.byref(c), 1, P(16), None, P(16), 1, P(256), None) == 1
    assert lib.msa_index_score(ctypes.byref(c), P(256), None, P(16), P(16), None) == 1
    assert lib.msa_index_score(ctypes.byref(c), P(256), P(18), P(16), P(16), None) == 1
    assert lib.msa_sparse_decode(ctypes.byref(c), P(256), P(16), None, P(16), P(16), None) == 1
    assert lib.msa_combine(ctypes.byref(c), P(256), P(4), P(16), None) == 1
    bad = _cfg(head_dim=64)
    assert lib.msa_topk_select(ctypes.byref(bad), P(256), P(16), P(16), None) == 2
    assert lib.msa_check_device_error(None, None, None) == 1
    assert lib.msa_noalloc_check_device_error(None, None) == 1


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "_lib", None)
    monkeypatch.setattr(ops, "_LIB_PATH", str(tmp_path / "libmsa.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ops.lib()
