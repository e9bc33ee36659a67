"""CPU-only checks of the C-ABI library: it builds, loads, exports every entry
point the header declares, and its host logic (split choice, workspace sizes,
argument validation) behaves as documented. No call here reaches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "streamkl.h")


@pytest.fixture(scope="module")
def lib():
    from attention_kl_loss_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(streamkl_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["streamkl_fwd", "streamkl_bwd", "streamkl_workspace_size",
                     "streamkl_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(["OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA",
                                 "ERR_TIMEOUT", "ERR_DEVICE_CHECK"]):
        assert lib.streamkl_status_string(code).decode() == "STREAMKL_" + name


def test_status_codes_agree_across_header_binding_and_kernels():
    """The device-side status codes (ptx.cuh), the header's enum and the
    binding's constants name the same numbers."""
    from attention_kl_loss_gb300 import binding
    text = open(HEADER).read()
    enum = dict((n, int(v)) for n, v in re.findall(r"(STREAMKL_\w+)\s*=\s*(\d+)", text))
    for name in ("STREAMKL_ERR_INVALID_ARG", "STREAMKL_ERR_TIMEOUT", "STREAMKL_ERR_DEVICE_CHECK"):
        assert enum[name] == getattr(binding, name)
    ptx = open(os.path.join(ROOT, "attention_kl_loss_gb300", "csrc", "ptx.cuh")).read()
    dev = dict((n, int(v)) for n, v in re.findall(r"constexpr int (kStatus\w+) = (\d+);", ptx))
    assert dev == {"kStatusInvalidArg": enum["STREAMKL_ERR_INVALID_ARG"],
                   "kStatusTimeout": enum["STREAMKL_ERR_TIMEOUT"],
                   "kStatusDeviceCheck": enum["STREAMKL_ERR_DEVICE_CHECK"]}


def test_device_status_is_raised_with_its_name():
    """raise_on_device_status turns each device code into a named error (CPU
    tensor: the synchronise is skipped on a host tensor)."""
    import torch
    from attention_kl_loss_gb300 import binding
    orig = torch.cuda.synchronize
    try:
        torch.cuda.synchronize = lambda *a, **k: None
        for code, name in [(4, "TIMEOUT"), (5, "DEVICE_CHECK"), (1, "INVALID_ARG")]:
            with pytest.raises(binding.StreamKLError) as e:
                binding.raise_on_device_status(torch.tensor([code], dtype=torch.int32), "test")
            assert e.value.status == code and f"STREAMKL_ERR_{name}" in str(e.value)
        binding.raise_on_device_status(torch.tensor([0], dtype=torch.int32), "test")
    finally:
        torch.cuda.synchronize = orig


def test_debug_build_exports_every_declared_symbol():
    """The debug build (device-side range checks) builds from the same sources
    and exports the same entry points; the binding can route its calls to it."""
    from attention_kl_loss_gb300 import binding, build
    path = build.build(debug=True)
    assert path.endswith("libstreamkl_debug.so") and os.path.exists(path)
    dbg = binding.load(debug=True)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.streamkl_status_string(5).decode() == "STREAMKL_ERR_DEVICE_CHECK"
    rel = binding.load(debug=False)
    assert dbg is not rel
    with binding.use_debug_library() as lib:
        assert lib is dbg and binding.load() is dbg
    assert binding.load() is rel


def test_split_choice(lib):
    # 128 (b,h) x 4 query tiles over 1024 key tiles: compute-bound, 3.4 waves
    # without a split; splitting the keys evens out the last wave
    assert lib.streamkl_choose_splits(4, 32, 512, 131072, 128, 1) > 1
    # plenty of query tiles: no split
    assert lib.streamkl_choose_splits(1, 32, 65536, 65536, 128, 1) == 1
    assert lib.streamkl_choose_splits(2, 16, 4096, 4096, 128, 0) == 1
    assert lib.streamkl_choose_splits(1, 8, 16384, 16384, 64, 0) == 1
    # one query row, 32 heads: 32 CTAs cannot stream K at full bandwidth, so
    # the keys are split across more SMs
    assert lib.streamkl_choose_splits(1, 32, 1, 65536, 128, 1) > 1
    # few query rows over 128 heads: already memory-bound with one CTA per
    # head (measured: splits 0.95-1.00x), so no split
    assert lib.streamkl_choose_splits(4, 32, 1, 65536, 128, 1) == 1
    assert lib.streamkl_choose_splits(4, 32, 64, 65536, 128, 1) == 1
    # invalid sizes
    assert lib.streamkl_choose_splits(1, 1, 8, 4, 64, 1) == 0


def test_workspace_sizes(lib):
    s = lib.streamkl_choose_splits(4, 32, 512, 131072, 128, 1)
    assert lib.streamkl_fwd_workspace_size(4, 32, 512, 131072, 128, 1, 0) == 5 * s * 128 * 512 * 4
    assert lib.streamkl_fwd_workspace_size(4, 32, 512, 131072, 128, 1, 1) == 0
    try:
        assert lib.streamkl_set_bwd_algorithm(1) == 0  # fused: fp32 dQ accumulators
        assert lib.streamkl_bwd_algorithm(1, 32, 65536, 65536, 128, 1, 1) == 1
        assert lib.streamkl_bwd_workspace_size(1, 32, 65536, 65536, 128, 1, 1) == 2 * 32 * 65536 * 128 * 4
        # one set under the per-key-tile fused kernel may be configuration 2
        # alone, which runs the separate kernels: room for their dQ partials too
        dq1 = lib.streamkl_bwd_dq_splits(1, 32, 65536, 65536, 128, 1, 0)
        assert lib.streamkl_bwd_workspace_size(1, 32, 65536, 65536, 128, 1, 0) == max(
            32 * 65536 * 128 * 4, dq1 * 32 * 65536 * 128 * 4 if dq1 > 1 else 0)
        dq = lib.streamkl_bwd_dq_splits(4, 32, 512, 131072, 128, 1, 0)
        dq_ws = dq * 128 * 512 * 128 * 4 if dq > 1 else 0
        assert lib.streamkl_workspace_size(4, 32, 512, 131072, 128, 1, 0) == max(
            5 * s * 128 * 512 * 4, 128 * 512 * 128 * 4, dq_ws)
        # the short-sweep kernel takes either set alone: one accumulator
        assert lib.streamkl_bwd_workspace_size(2, 8, 64, 65536, 128, 1, 0) == 2 * 8 * 64 * 128 * 4
        # separate: only the dQ kernel's key-split partials
        assert lib.streamkl_set_bwd_algorithm(0) == 0
        assert lib.streamkl_bwd_algorithm(1, 32, 65536, 65536, 128, 1, 1) == 0
        assert lib.streamkl_bwd_workspace_size(1, 32, 65536, 65536, 128, 1, 1) == 0
        dq = lib.streamkl_bwd_dq_splits(4, 32, 512, 131072, 128, 1, 0)
        dq_ws = dq * 128 * 512 * 128 * 4 if dq > 1 else 0
        assert lib.streamkl_bwd_workspace_size(4, 32, 512, 131072, 128, 1, 0) == dq_ws
        assert lib.streamkl_workspace_size(4, 32, 512, 131072, 128, 1, 0) == max(
            5 * s * 128 * 512 * 4, dq_ws)
        assert lib.streamkl_set_bwd_algorithm(7) == -1
    finally:
        lib.streamkl_set_bwd_algorithm(-1)


def test_automatic_backward_choice(lib):
    lib.streamkl_set_bwd_algorithm(-1)
    # separate kernels unless the query rows fit the fused short-sweep kernel
    # (at most 64 at d = 128) or, with one gradient set, a CTA of the fused
    # per-key-tile kernel sweeps enough query rows: 512 at d = 64, at d = 128
    # 512 without the mask and 1,024 with it
    for args in [(1, 32, 65536, 65536, 128, 1, 1), (4, 32, 65, 65536, 128, 1, 0),
                 (4, 32, 512, 131072, 128, 1, 0), (4, 32, 256, 65536, 128, 1, 0),
                 (4, 32, 1023, 65536, 128, 1, 0), (4, 32, 256, 8192, 128, 0, 0),
                 (2, 16, 4096, 4096, 128, 0, 1), (4, 32, 256, 65536, 64, 1, 0),
                 (4, 32, 64, 65536, 64, 1, 0), (1, 8, 16384, 16384, 64, 0, 1)]:
        assert lib.streamkl_bwd_algorithm(*args) == 0, args
    for args in [(4, 32, 64, 65536, 128, 1, 0), (1, 8, 1, 4096, 128, 0, 1),
                 (2, 2, 17, 300, 128, 1, 1), (4, 32, 512, 131072, 64, 1, 0),
                 (1, 8, 16384, 16384, 64, 0, 0), (2, 16, 4096, 4096, 128, 0, 0),
                 (4, 32, 512, 2048, 128, 0, 0), (4, 32, 1024, 65536, 128, 1, 0)]:
        assert lib.streamkl_bwd_algorithm(*args) == 1, args


def test_forward_pair_choice(lib):
    """CTA pairs only when switched on, and then for dense forwards without a
    split and an even number of 128-row query blocks."""
    assert lib.streamkl_fwd_pairs(1, 32, 65536, 65536, 128, 1, 0) == 0  # off by default
    try:
        assert lib.streamkl_set_fwd_pairs(1) == 0
        assert lib.streamkl_fwd_pairs(1, 32, 65536, 65536, 128, 1, 0) == 1
        assert lib.streamkl_fwd_pairs(2, 16, 4096, 4096, 128, 0, 0) == 1
        assert lib.streamkl_fwd_pairs(1, 2, 200, 300, 64, 1, 0) == 1   # two blocks, ragged
        assert lib.streamkl_fwd_pairs(1, 2, 300, 300, 64, 1, 0) == 0   # three blocks
        assert lib.streamkl_fwd_pairs(1, 2, 64, 300, 64, 1, 0) == 0    # one block
        assert lib.streamkl_fwd_pairs(4, 32, 512, 131072, 128, 1, 0) == 0  # split keys
        assert lib.streamkl_fwd_pairs(4, 32, 512, 131072, 128, 1, 1) == 1  # forced no split
        assert lib.streamkl_fwd_pairs(1, 1, 8, 4, 64, 1, 0) == -1
        assert lib.streamkl_set_fwd_pairs(3) == -1
    finally:
        lib.streamkl_set_fwd_pairs(0)


def test_dq_key_split_choice(lib):
    """The separate backward's dQ kernel splits its keys only when there are
    few query blocks: never at 64K (16,384 dQ CTAs), at least 2 ways for the
    split-K shape (512 CTAs, 3.4 waves on 152 SMs) and for one query block per
    head; the split partials' workspace follows the count, forced or not."""
    lib.streamkl_set_bwd_dq_splits(0)
    assert lib.streamkl_bwd_dq_splits(1, 32, 65536, 65536, 128, 1, 1) == 1
    assert lib.streamkl_bwd_dq_splits(4, 32, 512, 131072, 128, 1, 0) >= 2
    assert lib.streamkl_bwd_dq_splits(1, 4, 128, 131072, 128, 1, 0) >= 8
    assert lib.streamkl_bwd_dq_splits(1, 1, 8, 4, 64, 1, 0) == -1  # invalid sizes
    try:
        assert lib.streamkl_set_bwd_dq_splits(3) == 0
        # 200 keys = 4 steps of 64: 3 requested -> 2 steps each -> 2 splits
        assert lib.streamkl_bwd_dq_splits(1, 1, 100, 200, 64, 0, 0) == 2
        assert lib.streamkl_bwd_workspace_size(1, 1, 100, 200, 64, 0, 0) == 2 * 100 * 64 * 4
        assert lib.streamkl_bwd_workspace_size(1, 1, 100, 200, 64, 0, 1) == 2 * 2 * 100 * 64 * 4
        assert lib.streamkl_bwd_dq_splits(1, 1, 8, 8, 64, 0, 0) == 1  # one step: no split
        assert lib.streamkl_bwd_workspace_size(1, 1, 8, 8, 64, 0, 0) == 0
        assert lib.streamkl_set_bwd_dq_splits(-1) == -1
    finally:
        lib.streamkl_set_bwd_dq_splits(0)


def test_persistent_dk_choice(lib):
    """The persistent dK kernel is used for short query sweeps (N_Q <= 384)
    with more (key block, batch-head) items than SMs, one CTA per SM; the
    override forces or disables it."""
    lib.streamkl_set_bwd_dk_persist(0)
    sms = lib.streamkl_bwd_dk_persist(4, 32, 384, 131072, 128, 1)
    assert sms > 0  # 1024 key blocks x 128 slices
    assert lib.streamkl_bwd_dk_persist(4, 32, 64, 65536, 128, 1) == sms
    # 8 query steps per key block (the split-K shape): one CTA per key block
    assert lib.streamkl_bwd_dk_persist(4, 32, 512, 131072, 128, 1) == 0
    assert lib.streamkl_bwd_dk_persist(4, 32, 1024, 65536, 128, 1) == 0
    assert lib.streamkl_bwd_dk_persist(1, 32, 65536, 65536, 128, 1) == 0
    assert lib.streamkl_bwd_dk_persist(1, 1, 512, 512, 64, 0) == 0  # 4 items: fewer than SMs
    assert lib.streamkl_bwd_dk_persist(1, 1, 8, 4, 64, 1) == -1  # invalid sizes
    try:
        assert lib.streamkl_set_bwd_dk_persist(3) == 0
        assert lib.streamkl_bwd_dk_persist(1, 32, 65536, 65536, 128, 1) == 3
        assert lib.streamkl_set_bwd_dk_persist(-1) == 0
        assert lib.streamkl_bwd_dk_persist(4, 32, 384, 131072, 128, 1) == 0
        assert lib.streamkl_set_bwd_dk_persist(-2) == -1
    finally:
        lib.streamkl_set_bwd_dk_persist(0)


def test_forced_split_workspace_rounding(lib):
    # 100 rows, 2 key tiles, request 16 splits -> 2 effective splits
    n = 5 * 2 * 1 * 100 * 4
    want = (n + 255) // 256 * 256
    assert lib.streamkl_fwd_workspace_size(1, 1, 100, 200, 64, 0, 16) == want


def _fwd(lib, q=0x1000, NQ=8, NK=8, d=64, causal=0, kl=0x2000, status=0x3000, scale=0.125):
    P = ctypes.c_void_p
    return lib.streamkl_fwd(P(q), P(q), P(q), P(q), 1, 1, NQ, NK, d, scale, causal, 0, P(kl),
                            P(kl), P(kl), None, 0, P(status), None)


def test_argument_validation_is_synchronous(lib):
    assert _fwd(lib, q=0) == 1  # NULL input
    assert b"q1" in lib.streamkl_last_error()
    assert _fwd(lib, q=0x1001) == 1  # misaligned
    assert _fwd(lib, d=96) == 2  # unsupported head dim
    assert _fwd(lib, NQ=16, NK=8, causal=1) == 1  # causal needs NQ <= NK
    assert _fwd(lib, kl=0) == 1
    assert _fwd(lib, status=0) == 1
    assert _fwd(lib, scale=0.0) == 1
    assert _fwd(lib, NQ=0) == 1


def test_backward_validation(lib):
    P = ctypes.c_void_p
    a = P(0x1000)

    def bwd(dq1, dk1, ws=0x4000, ws_bytes=1 << 20):
        return lib.streamkl_bwd(a, a, a, a, 1, 1, 8, 8, 64, 0.125, 0, a, a, a, a, a, a,
                                P(dq1) if dq1 else None, P(dk1) if dk1 else None,
                                P(ws) if ws else None, ws_bytes, a, None)

    assert bwd(0x1000, 0) == 1  # dq1 without dk1
    assert bwd(0, 0x1000) == 1

    def bwd_sets(dq2, dk2, dq1, dk1):
        f = lambda v: P(v) if v else None
        return lib.streamkl_bwd(a, a, a, a, 1, 1, 8, 8, 64, 0.125, 0, a, a, a, a, f(dq2), f(dk2),
                                f(dq1), f(dk1), None, 0, None, None)

    assert bwd_sets(0, 0, 0, 0) == 1  # no gradient at all
    assert b"no gradient" in lib.streamkl_last_error()
    assert bwd_sets(0x1000, 0, 0x1000, 0x1000) == 1  # dq2 without dk2
    # configuration 2 alone passes the gradient checks and fails only on the
    # missing status word (checked last)
    assert bwd_sets(0, 0, 0x1000, 0x1000) == 1
    assert b"dev_status" in lib.streamkl_last_error()
    try:
        lib.streamkl_set_bwd_algorithm(1)  # the fused algorithm needs a workspace
        assert bwd(0, 0, ws=0) == 1
        assert bwd(0, 0, ws_bytes=16) == 1
        assert b"workspace" in lib.streamkl_last_error()
    finally:
        lib.streamkl_set_bwd_algorithm(-1)


def test_reverse_direction_validation(lib):
    """The reverse entry points check their own gradient pairs by their own
    names and otherwise fail exactly like the exchanged forward/backward call."""
    P = ctypes.c_void_p
    a = P(0x1000)
    f = lambda v: P(v) if v else None

    def fwd_rev(q1=0x1000, q2=0x1000, d=64, NQ=8, NK=8, causal=0):
        return lib.streamkl_fwd_reverse(f(q1), a, f(q2), a, 1, 1, NQ, NK, d, 0.125, causal, 0, a,
                                        a, a, None, 0, a, None)

    assert fwd_rev(q2=0) == 1
    assert b"q1" in lib.streamkl_last_error()  # named by its slot in the exchanged call
    assert fwd_rev(q1=0x1001) == 1  # misaligned
    assert fwd_rev(d=96) == 2
    assert fwd_rev(NQ=16, NK=8, causal=1) == 1

    def bwd_rev(dq2, dk2, dq1, dk1, status=None, ws=None, ws_bytes=0):
        return lib.streamkl_bwd_reverse(a, a, a, a, 1, 1, 8, 8, 64, 0.125, 0, a, a, a, a, f(dq2),
                                        f(dk2), f(dq1), f(dk1), f(ws), ws_bytes, f(status), None)

    assert bwd_rev(0x1000, 0, 0, 0) == 1
    assert b"dq2 and dk2" in lib.streamkl_last_error()
    assert bwd_rev(0, 0, 0, 0x1000) == 1
    assert b"dq1 and dk1" in lib.streamkl_last_error()
    assert bwd_rev(0, 0, 0, 0) == 1
    assert b"no gradient" in lib.streamkl_last_error()
    # the student's gradients alone pass every check but the missing status word
    assert bwd_rev(0x1000, 0x1000, 0, 0) == 1
    assert b"dev_status" in lib.streamkl_last_error()
    try:
        lib.streamkl_set_bwd_algorithm(1)
        # with the teacher's gradients the fused algorithm needs its workspace
        assert bwd_rev(0x1000, 0x1000, 0x1000, 0x1000, status=0x3000) == 1
        assert b"workspace" in lib.streamkl_last_error()
    finally:
        lib.streamkl_set_bwd_algorithm(-1)


def test_selftest_validation(lib):
    assert lib.streamkl_selftest_wait_timeout(None, 100, None) == 1
    assert lib.streamkl_selftest_wait_timeout(ctypes.c_void_p(0x1000), 0, None) == 1


def test_pair_counts():
    from attention_kl_loss_gb300 import synthetic
    w = synthetic.WORKLOADS["causal64k"]
    assert w.live_pairs_per_head() == 65536 * 65537 // 2
    w4 = synthetic.WORKLOADS["splitk"]
    brute = sum(i + 1 + (131072 - 512) for i in range(512))
    assert w4.live_pairs_per_head() == brute


def test_packed_batch_validation(lib):
    """Host checks of the variable-length entry points (the offsets are device
    data and are checked by the kernels)."""
    P = ctypes.c_void_p
    a, cu = P(0x1000), P(0x2000)

    def fwd(cu_q=cu, cu_k=cu, total_q=300, total_k=400, max_q=200, max_k=250, d=64):
        return lib.streamkl_fwd_varlen(a, a, a, a, cu_q, cu_k, 2, 4, total_q, total_k, max_q, max_k,
                                       d, 0.125, 1, a, a, a, a, None)

    assert fwd(cu_q=None) == 1
    assert b"cu_seqlens" in lib.streamkl_last_error()
    assert fwd(cu_q=P(0x2002)) == 1  # misaligned offsets
    assert fwd(max_q=301) == 1  # longer than the packed total
    assert fwd(total_k=0) == 1
    assert fwd(d=96) == 2
    st = lib.streamkl_bwd_varlen(a, a, a, a, cu, cu, 2, 4, 300, 400, 200, 250, 64, 0.125, 1, a, a,
                                 a, a, None, None, None, None, a, None)
    assert st == 1 and b"no gradient" in lib.streamkl_last_error()
