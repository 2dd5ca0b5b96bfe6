"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host (no GPU needed: nothing here launches a kernel)."""

import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dm():
    import __graft_entry__

    __graft_entry__.build()
    import decode_context_mla_causal_gb300 as mod

    return mod


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(dcp_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_three_steps():
    names = _declared_functions()
    for n in ("dcp_mla_metadata", "dcp_mla_partial", "dcp_lse_merge"):
        assert n in names


def test_every_declared_symbol_is_exported(dm):
    lib = ctypes.CDLL(dm.library_path())
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_subpage_size_matches_golden(dm):
    import json

    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "subpage_review.json")))["cases"]
    for bs, want in cases:
        assert dm.dcp_mla_subpage_size(bs) == want
    assert dm.dcp_mla_subpage_size(0) == -1


def _dims(dm, **kw):
    base = dict(batch=2, qlen=3, num_heads=8, dcp=2, interleave=1, block_size=16,
                max_blocks_per_seq=8, max_local_len=100, num_blocks=64, num_splits=2)
    base.update(kw)
    return dm.make_dims(**base)


@pytest.mark.parametrize("bad", [
    dict(qlen=0), dict(num_heads=0), dict(dcp=0), dict(interleave=0), dict(interleave=32),
    dict(interleave=3), dict(block_size=0), dict(max_local_len=-1), dict(max_blocks_per_seq=2),
    dict(num_blocks=0), dict(num_splits=0), dict(batch=-1), dict(causal=2),
    dict(base_splits=-1), dict(base_splits=3),
])
def test_invalid_dims_rejected_before_launch(dm, bad):
    d = _dims(dm, **{k: v for k, v in bad.items() if k != "causal"})
    if "causal" in bad:
        d.causal = bad["causal"]
    with pytest.raises(dm.DcpError) as ei:
        dm.dcp_mla_check_dims(d)
    assert ei.value.code == dm.DCP_ERR_INVALID_ARG
    assert dm.dcp_last_error()


def test_base_splits_range(dm):
    # 0 and num_splits both mean "no balancing"; anything between turns it on
    for base in (0, 1, 2):
        dm.dcp_mla_check_dims(_dims(dm, num_splits=2, base_splits=base))
    # balancing reads every (rank, sequence) pair's length in each metadata CTA
    d = _dims(dm, batch=1 << 14, dcp=8, num_splits=2, base_splits=1)
    with pytest.raises(dm.DcpError) as ei:
        dm.dcp_mla_check_dims(d)
    assert ei.value.code == dm.DCP_ERR_UNSUPPORTED


def test_concurrent_items_without_a_device(dm):
    import torch

    if torch.cuda.is_available():
        assert dm.dcp_mla_concurrent_items() >= 1
    else:
        assert dm.dcp_mla_concurrent_items() == -1
        assert "CUDA device" in dm.dcp_last_error()  # the failure says why


def test_rank_range_checked(dm):
    d = _dims(dm)
    lib = dm.load()
    assert lib.dcp_mla_check_dims(ctypes.byref(d), 0, 2) == dm.DCP_OK
    assert lib.dcp_mla_check_dims(ctypes.byref(d), 1, 2) == dm.DCP_ERR_INVALID_ARG
    assert lib.dcp_mla_check_dims(ctypes.byref(d), -1, 1) == dm.DCP_ERR_INVALID_ARG


def test_null_pointers_rejected_without_launch(dm):
    d = _dims(dm)
    lib = dm.load()
    rc = lib.dcp_mla_metadata(ctypes.byref(d), None, None, 0, 2, None, None, None, None,
                              None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG
    rc = lib.dcp_mla_partial(ctypes.byref(d), None, None, 1, None, 0.1, 0, 2, None, None,
                             None, None, None, None, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG
    rc = lib.dcp_lse_merge(ctypes.byref(d), 2, None, None, None, None, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG
    rc = lib.dcp_mla_partial(ctypes.byref(d), None, None, 7, None, 0.1, 0, 2, None, None,
                             None, None, None, None, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "kv_dtype" in dm.dcp_last_error()


def test_empty_batch_is_a_no_op(dm):
    d = _dims(dm, batch=0)
    lib = dm.load()
    assert lib.dcp_mla_metadata(ctypes.byref(d), None, None, 0, 2, None, None, None, None,
                                None, None) == dm.DCP_OK


def test_max_pages(dm):
    assert dm.dcp_mla_max_pages(_dims(dm, max_local_len=100, block_size=16)) == 7
    assert dm.dcp_mla_max_pages(_dims(dm, max_local_len=131072, block_size=64,
                                      max_blocks_per_seq=2048)) == 2048
    assert dm.dcp_mla_max_pages(_dims(dm, max_local_len=300, block_size=96,
                                      max_blocks_per_seq=4)) == 10


def test_a2a_chunk_words_and_argument_checks(dm):
    lib = dm.load()
    d = _dims(dm, batch=4, qlen=3, num_heads=128, dcp=8, block_size=64, max_blocks_per_seq=2048,
              max_local_len=131072)
    # 12 rows x 16 heads x (512 outputs + 2 LSE words), already a multiple of 8
    assert dm.dcp_a2a_chunk_words(d) == 12 * 16 * 514
    assert dm.dcp_a2a_chunk_words(d, 128) == 12 * 16 * 130
    small = _dims(dm, batch=1, qlen=3, num_heads=2, dcp=2)  # 3 x 1 x 2 LSE words -> padded
    assert dm.dcp_a2a_chunk_words(small) == 3 * 512 + 8
    assert lib.dcp_a2a_chunk_words(ctypes.byref(_dims(dm, num_heads=6, dcp=4)), 512) == -1
    assert lib.dcp_a2a_chunk_words(ctypes.byref(d), 0) == -1
    # the projected payload is a multiple of 16 in [16, 256]
    rc = lib.dcp_a2a_project(ctypes.byref(d), 8, None, None, 100, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "multiple of 16" in dm.dcp_last_error()
    rc = lib.dcp_a2a_project(ctypes.byref(d), 8, None, None, 128, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "NULL" in dm.dcp_last_error()
    rc = lib.dcp_a2a_pack(ctypes.byref(d), 8, None, None, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "NULL" in dm.dcp_last_error()
    rc = lib.dcp_a2a_pack(ctypes.byref(_dims(dm, num_heads=6, dcp=4)), 4, None, None, None,
                          None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "multiple of dcp" in dm.dcp_last_error()
    rc = lib.dcp_a2a_combine(ctypes.byref(d), 512, None, 12, 0, 0, 1, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG and "strides" in dm.dcp_last_error()
    rc = lib.dcp_a2a_combine(ctypes.byref(d), 512, None, 8, 0, 7, 2, None, None, None, None)
    assert rc == dm.DCP_ERR_INVALID_ARG  # destinations beyond dcp


def test_workspace_size(dm):
    # one int32 per work item (rank, sequence, split, 128-row tile) and the count of
    # listed items, rounded up to a 16-byte multiple
    d = _dims(dm, batch=32, qlen=5, num_heads=128, dcp=8, num_splits=1)
    assert dm.dcp_mla_workspace_size(d, 8) == (8 * 32 * 1 * 5 + 1) * 4 + 12
    d = _dims(dm, batch=1, qlen=3, num_heads=8, dcp=2, num_splits=3)
    assert dm.dcp_mla_workspace_size(d, 1) == 16  # 3 items and the count
    lib = dm.load()
    assert lib.dcp_mla_workspace_size(ctypes.byref(d), 1, None) == dm.DCP_ERR_INVALID_ARG
