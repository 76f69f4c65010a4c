"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every symbol include/treewy.h declares, the ctypes structure matches the C
layout, and host-side validation rejects bad arguments before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from gdn_speculative_tree_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treewy.h")


@pytest.fixture(scope="module")
def lib():
    try:
        build.nvcc_path()
    except RuntimeError:
        pytest.skip("no CUDA toolkit")
    path = build.build()
    return binding.load(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(treewy_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in binding.ENTRY_POINTS:
        assert n in names
    assert set(names) <= set(binding.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert b"sm_103a" in lib.treewy_version()


def test_struct_layout_matches_c():
    # int32 x6, int64 x2, 13 pointers, uint32 x2 on an LP64 ABI
    assert ctypes.sizeof(binding.TreewyBatch) == 6 * 4 + 2 * 8 + 13 * 8 + 2 * 4
    assert binding.TreewyBatch.T.offset == 24
    assert binding.TreewyBatch.node_offset.offset == 40
    assert binding.TreewyBatch.flags.offset == 40 + 13 * 8


def _valid_batch():
    b = binding.TreewyBatch()
    b.R, b.H, b.dk, b.dv, b.max_nodes, b.qkv_dtype = 2, 4, 128, 128, 64, binding.DTYPE_BF16
    b.T, b.num_slots = 10, 2
    fake = 0x10000  # never dereferenced: these calls fail validation first
    for f in ("node_offset", "parent", "q", "k", "v", "alpha", "beta", "state", "state_slot",
              "o", "U", "status"):
        setattr(b, f, fake)
    return b


@pytest.mark.parametrize("field,value,code", [
    ("R", -1, binding.TREEWY_ERR_INVALID_ARG),
    ("H", 0, binding.TREEWY_ERR_INVALID_ARG),
    ("dk", 0, binding.TREEWY_ERR_INVALID_ARG),
    ("dk", 256, binding.TREEWY_ERR_UNSUPPORTED),
    ("dv", 129, binding.TREEWY_ERR_UNSUPPORTED),
    ("max_nodes", 65, binding.TREEWY_ERR_UNSUPPORTED),
    ("max_nodes", 0, binding.TREEWY_ERR_UNSUPPORTED),
    ("qkv_dtype", 7, binding.TREEWY_ERR_INVALID_ARG),
    ("T", -5, binding.TREEWY_ERR_INVALID_ARG),
    ("num_slots", 0, binding.TREEWY_ERR_INVALID_ARG),
    ("q", None, binding.TREEWY_ERR_INVALID_ARG),
    ("status", None, binding.TREEWY_ERR_INVALID_ARG),
    ("state", 0x10004, binding.TREEWY_ERR_INVALID_ARG),
    ("k", 0x10008, binding.TREEWY_ERR_INVALID_ARG),
    ("o", 0x10004, binding.TREEWY_ERR_INVALID_ARG),
    ("U", 0x10008, binding.TREEWY_ERR_INVALID_ARG),
])
def test_verify_rejects_bad_arguments(lib, field, value, code):
    b = _valid_batch()
    setattr(b, field, value)
    rc = lib.treewy_verify(ctypes.byref(b), None)
    assert rc == code
    assert lib.treewy_last_error().decode()


def test_null_batch_and_null_accepted(lib):
    assert lib.treewy_verify(None, None) == binding.TREEWY_ERR_INVALID_ARG
    b = _valid_batch()
    assert lib.treewy_commit(ctypes.byref(b), None, None) == binding.TREEWY_ERR_INVALID_ARG
    assert b"accepted" in lib.treewy_last_error()
    assert lib.treewy_storeall_verify(ctypes.byref(b), None, None) == binding.TREEWY_ERR_INVALID_ARG
    assert lib.treewy_storeall_commit(ctypes.byref(b), 0x10000, None, None) == \
        binding.TREEWY_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    b = binding.TreewyBatch()
    b.R, b.H, b.dk, b.dv, b.max_nodes, b.qkv_dtype, b.T, b.num_slots = 0, 1, 128, 128, 64, 0, 0, 1
    assert lib.treewy_verify(ctypes.byref(b), None) == binding.TREEWY_OK
    assert lib.treewy_commit(ctypes.byref(b), None, None) == binding.TREEWY_OK


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load(str(tmp_path / "nope.so"))


def test_commit_verify_rejects_inconsistent_rounds(lib):
    prev, nxt = _valid_batch(), _valid_batch()
    prev.R = 3
    assert lib.treewy_commit_verify(ctypes.byref(prev), 0x10000, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG
    assert b"same R" in lib.treewy_last_error()
    prev = _valid_batch()
    prev.state = 0x20000
    assert lib.treewy_commit_verify(ctypes.byref(prev), 0x10000, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG
    assert b"state pool" in lib.treewy_last_error()
    prev = _valid_batch()
    prev.U = 0x10004
    assert lib.treewy_commit_verify(ctypes.byref(prev), 0x10000, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG
    assert b"aligned" in lib.treewy_last_error()
    b = _valid_batch()
    b.U = 0x10004
    assert lib.treewy_commit(ctypes.byref(b), 0x10000, None) == binding.TREEWY_ERR_INVALID_ARG
    assert b"aligned" in lib.treewy_last_error()
    prev = _valid_batch()
    assert lib.treewy_commit_verify(ctypes.byref(prev), None, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG
    assert lib.treewy_commit_verify(None, 0x10000, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG


def test_state_flags(lib):
    b = _valid_batch()
    b.flags = 4  # no such flag
    assert lib.treewy_verify(ctypes.byref(b), None) == binding.TREEWY_ERR_INVALID_ARG
    assert b"unknown bits" in lib.treewy_last_error()
    b = _valid_batch()
    b.flags = binding.FLAG_STATE_BF16
    assert lib.treewy_storeall_verify(ctypes.byref(b), 0x10000, None) == binding.TREEWY_ERR_UNSUPPORTED
    assert lib.treewy_storeall_commit(ctypes.byref(b), 0x10000, 0x10000, None) == \
        binding.TREEWY_ERR_UNSUPPORTED
    prev, nxt = _valid_batch(), _valid_batch()
    nxt.flags = binding.FLAG_STATE_BF16
    assert lib.treewy_commit_verify(ctypes.byref(prev), 0x10000, ctypes.byref(nxt), None) == \
        binding.TREEWY_ERR_INVALID_ARG
    assert b"STATE_BF16" in lib.treewy_last_error()


def test_make_batch_sets_the_state_flag():
    torch = pytest.importorskip("torch")
    from gdn_speculative_tree_gb300 import workloads as wl
    w = wl.assemble([wl.chain_parents(3)], [1], 2, 16, 16, "bf16", 0.05, (0.9, 0.999), ("sigmoid",),
                    seed=1, state_dtype="bf16")
    assert w.state.dtype == torch.bfloat16
    o = torch.empty(w.T, w.H, w.dv)
    st = torch.zeros(w.R, dtype=torch.int32)
    b = binding.make_batch(node_offset=w.node_offset, parent=w.parent, q=w.q, k=w.k, v=w.v,
                           alpha=w.alpha, beta=w.beta, state=w.state, state_slot=w.state_slot,
                           o=o, U=o, status=st)
    assert b.flags == binding.FLAG_STATE_BF16
    w32 = wl.assemble([wl.chain_parents(3)], [1], 2, 16, 16, "bf16", 0.05, (0.9, 0.999),
                      ("sigmoid",), seed=1)
    assert torch.equal(w32.state.to(torch.bfloat16), w.state)  # same draw, rounded
    with pytest.raises(TypeError):
        binding.make_batch(node_offset=w.node_offset, parent=w.parent, q=w.q, k=w.k, v=w.v,
                           alpha=w.alpha, beta=w.beta, state=w.state.half(),
                           state_slot=w.state_slot, o=o, U=o, status=st)


def test_too_many_request_head_pairs(lib):
    b = _valid_batch()
    b.R, b.H = 1 << 20, 1 << 12
    assert lib.treewy_verify(ctypes.byref(b), None) == binding.TREEWY_ERR_UNSUPPORTED
    assert b"R * H" in lib.treewy_last_error()


def test_wait_selftest_validates_before_launch(lib):
    # rejected on the host: no status word, a misaligned one, limits outside 1 .. 1e7 us
    assert lib.treewy_selftest_wait_timeout(None, 1000, None) == binding.TREEWY_ERR_INVALID_ARG
    assert lib.treewy_selftest_wait_timeout(0x10002, 1000, None) == binding.TREEWY_ERR_INVALID_ARG
    assert lib.treewy_selftest_wait_timeout(0x10000, 0, None) == binding.TREEWY_ERR_INVALID_ARG
    assert lib.treewy_selftest_wait_timeout(0x10000, 10_000_001, None) == binding.TREEWY_ERR_INVALID_ARG
    assert "limit_us" in lib.treewy_last_error().decode()
