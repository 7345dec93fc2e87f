"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/sdm.h declares, and rejects bad arguments on the host (no GPU needed:
these paths return before any CUDA call)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from speculative_decoding_markov_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdm_[a-z_]+)\s*\(", text)))


def test_header_declares_the_five_operations():
    names = declared_functions()
    for op in ("sdm_draft_chain", "sdm_draft_tree", "sdm_schedule_budget", "sdm_pack_ragged", "sdm_verify"):
        assert op in names
    assert set(names) == set(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.sdm_status_str(0) == b"ok"
    assert lib.sdm_status_str(5) == b"workspace missing or too small"
    assert lib.sdm_version() >= 100


def test_timeout_check_host_validation(lib):
    f = lib.sdm_check_timeout_path
    a = [FAKE, 0, FAKE, FAKE, FAKE, 4, 7, 1024, 64, 50_000, FAKE, 1 << 30, FAKE, None]
    bad = list(a)
    bad[9] = 10                                 # a limit below 1 us
    assert f(*bad) == 1
    bad[9] = 2_000_000_000                      # above 1 s
    assert f(*bad) == 1
    bad = list(a)
    bad[12] = None                              # the status word is where the result goes
    assert f(*bad) == 1
    bad = list(a)
    bad[11] = 16                                # workspace too small
    assert f(*bad) == 5


def test_device_bits_map_to_a_status(lib):
    f = lib.sdm_status_of_device
    assert f(0) == 0
    assert f(binding.DEV_TIER_UNCAPTURED) == 0                     # informational: run uncaptured
    assert f(binding.DEV_TIER_OVERFLOW) == 3                       # SDM_ERR_TIER_OVERFLOW (strict pack)
    assert f(binding.DEV_TIER_OVERFLOW | binding.DEV_TIER_UNCAPTURED) == 3
    assert f(binding.DEV_TIMEOUT | binding.DEV_TIER_OVERFLOW) == 7   # a timed-out wait comes first
    for bit in (binding.DEV_BAD_TOKEN, binding.DEV_BAD_WINDOW, binding.DEV_CAPACITY, binding.DEV_BAD_CLASS):
        assert f(bit) == 6                                         # SDM_ERR_DEVICE
    assert lib.sdm_status_str(3) == b"packed total above every tier"
    assert lib.sdm_status_str(7) == b"a bounded device wait ran out"


def test_workspace_sizes_are_host_computable(lib):
    assert lib.sdm_workspace_size(binding.OP_DRAFT_CHAIN, 64, 7, 151936, 256, 0, 0, 0) > 0
    assert lib.sdm_workspace_size(binding.OP_DRAFT_TREE, 32, 16, 151936, 256, 8, 4, 64) > 0
    assert lib.sdm_workspace_size(binding.OP_VERIFY, 64, 7, 151936, 256, 512, 0, 0) >= 512 * 8
    assert lib.sdm_workspace_size(binding.OP_VERIFY_TREE, 32, 16, 151936, 0, 0, 0, 64) >= 32 * 65 * 8
    assert lib.sdm_workspace_size(binding.OP_SCHEDULE, 64, 7, 0, 0, 0, 0, 0) == 0


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first


def _chain(lib, **kw):
    a = dict(L=FAKE, dtL=0, U=FAKE, W=FAKE, anchor=FAKE, R=4, B=7, V=1024, r=64, dec=0, T=1.0, tokens=FAKE,
             ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.sdm_draft_chain(a["L"], a["dtL"], a["U"], a["W"], None, a["anchor"], a["R"], a["B"], a["V"], a["r"],
                               a["dec"], a["T"], binding.SdmRng(0, 0), a["tokens"], None, None, a["ws"],
                               a["ws_bytes"], None, None)


def test_draft_chain_host_validation(lib):
    assert _chain(lib, L=None) == 1
    assert _chain(lib, R=0) == 1
    assert _chain(lib, dtL=7) == 1
    assert _chain(lib, dec=1, T=0.0) == 1
    assert _chain(lib, V=1001) == 2            # V % 8 != 0
    assert _chain(lib, r=96) == 2              # r % 64 != 0
    assert _chain(lib, r=512) == 2             # r > 256
    assert _chain(lib, L=ctypes.c_void_p(0x1004)) == 2   # misaligned base
    assert _chain(lib, ws=None) == 5
    assert _chain(lib, ws_bytes=16) == 5
    assert _chain(lib, dec=1, V=524288 + 8) == 2   # sampling: the draw's chunk table holds 32768 records


def _front(lib, **kw):
    a = dict(L=FAKE, dtL=0, prepared=FAKE, R=64, B=7, V=1024, r=64, use_budget=1, tiers=FAKE, n_tiers=2, strict=0,
             capacity=1024, ws=FAKE, ws_bytes=1 << 30)
    a.update(kw)
    return lib.sdm_draft_chain_front(a["L"], a["dtL"], FAKE, FAKE, a["prepared"], FAKE, a["R"], a["B"], a["V"], a["r"],
                                     FAKE, FAKE, a["use_budget"], a["tiers"], a["n_tiers"], a["strict"], FAKE, FAKE,
                                     FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["capacity"], FAKE, FAKE, a["ws"],
                                     a["ws_bytes"], None, None)


def test_draft_chain_front_host_validation(lib):
    assert _front(lib, prepared=None) == 1      # the bound-pruned chain needs the prepared tables
    assert _front(lib, strict=2) == 1
    assert _front(lib, use_budget=2) == 1
    assert _front(lib, tiers=None) == 1         # tiers missing
    assert _front(lib, capacity=0) == 1
    assert _front(lib, V=1001) == 2             # V % 8 != 0
    assert _front(lib, R=2000, B=8) == 2        # R * B > 8192: the scheduler ranks in shared memory
    assert _front(lib, R=512, B=8) == 2         # R * B = 4096: the scheduler's arrays exceed 48 KB
    assert _front(lib, B=65) == 2               # more steps than the pick walks
    assert _front(lib, ws_bytes=16) == 5
    assert lib.sdm_workspace_size(binding.OP_DRAFT_CHAIN, 64, 7, 1024, 64, 0, 0, 0) <= 1 << 30


def test_prepare_host_validation(lib):
    assert lib.sdm_markov_prepared_size(151936, 256) >= 151936 * 256 * 2 + 3 * 151936 * 4
    assert lib.sdm_markov_prepare(None, FAKE, 1024, 64, FAKE, 1 << 30, None, None) == 1
    assert lib.sdm_markov_prepare(FAKE, FAKE, 1020, 64, FAKE, 1 << 30, None, None) == 2
    assert lib.sdm_markov_prepare(FAKE, FAKE, 1024, 64, FAKE, 16, None, None) == 5


def test_tree_and_verify_host_validation(lib):
    f = lib.sdm_draft_tree
    # L, dtL, U, W, prepared, anchor, R, B, V, r, k, P, N, outputs x 6, ws, ws_bytes, dev_status, stream
    args = [FAKE, 0, FAKE, FAKE, None, FAKE, 32, 16, 1024, 64, 4, 8, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
            1 << 30, None, None]
    bad_k = list(args)
    bad_k[10] = 9                               # k > 8
    assert f(*bad_k) == 2
    bad_p = list(args)
    bad_p[11] = 3                               # 128 % P != 0
    assert f(*bad_p) == 2
    bad_n = list(args)
    bad_n[12] = 8 * 16 + 1                      # N > P * B
    assert f(*bad_n) == 2
    big_pool = list(args)
    big_pool[7], big_pool[11], big_pool[10] = 128, 64, 1   # P * B + 1 > 8192 (pool ranked in shared memory)
    assert f(*big_pool) == 2
    big_v = list(args)
    big_v[8] = 524288 + 8                       # V beyond the level select's chunk and candidate tables
    assert f(*big_v) == 2
    small_ws = list(args)
    small_ws[20] = 1024                         # the workspace holds the scan lists or the records
    assert f(*small_ws) == 5
    bad_prep = list(args)
    bad_prep[4] = ctypes.c_void_p(0x1008)       # prepared tables must be 16-byte aligned
    assert f(*bad_prep) == 2
    # the tree's workspace covers both level paths
    assert lib.sdm_workspace_size(binding.OP_DRAFT_TREE, 32, 16, 151936, 256, 8, 4, 64) >= 32 * 16 * 10 * 512 * 8
    vt = lib.sdm_verify_tree
    assert vt(FAKE, 0, FAKE, FAKE, FAKE, 4, 16384, 7, 1024, FAKE, FAKE, FAKE, FAKE, 1 << 30, None, None) == 2
    v = lib.sdm_verify
    vargs = [2, 0, 1.0, binding.SdmRng(0, 0), FAKE, 0, 64, FAKE, FAKE, FAKE, None, None, None, None, 0, None, None, 0,
             4, 7, 1024, FAKE, None, FAKE, FAKE, FAKE, 1 << 30, None, None]
    assert v(*vargs) == 1                       # cap-accept without a budget
    vargs[0] = 1
    vargs[1] = 1                                # sample without logq / L / U / W
    assert v(*vargs) == 1
    assert lib.sdm_schedule_budget(FAKE, 2000, 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None, None) == 2
    sd = lib.sdm_schedule_dynamic
    assert sd(FAKE, None, 4, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 1   # no stale confidences
    assert sd(FAKE, FAKE, 2000, 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 2   # R * gamma > 8192
    assert lib.sdm_pack_ragged(FAKE, FAKE, None, 4, 7, None, 2, 0, FAKE, FAKE, FAKE, FAKE, 64, FAKE, None, None,
                               None) == 1       # tiers missing
    assert lib.sdm_pack_ragged(FAKE, FAKE, None, 4, 7, FAKE, 2, 2, FAKE, FAKE, FAKE, FAKE, 64, FAKE, None, None,
                               None) == 1       # strict is 0 or 1


def test_observability_host_validation(lib):
    # tv_label: workspace holds the target LSE partials, the row list and the GEMM partials
    n = lib.sdm_workspace_size(binding.OP_TV_LABEL, 256, 16, 151936, 256, 4352, 0, 0)
    assert n >= 4352 * 10 * 8 + 6 * 4096 * 4 + 4096 * 4 * 8
    tv = lib.sdm_tv_label
    a = [1.0, FAKE, 0, 64, FAKE, FAKE, FAKE, None, FAKE, 0, FAKE, FAKE, 64, 4, 7, 1024, FAKE, FAKE, 1 << 30, None, None]
    bad = list(a)
    bad[0] = 0.0                                # temperature must be positive
    assert tv(*bad) == 1
    bad = list(a)
    bad[8] = None                               # L missing
    assert tv(*bad) == 1
    bad = list(a)
    bad[15] = 1020                              # V % 8 != 0
    assert tv(*bad) == 2
    bad = list(a)
    bad[12] = 96                                # r % 64 != 0
    assert tv(*bad) == 2
    bad = list(a)
    bad[18] = 16                                # workspace too small
    assert tv(*bad) == 5
    ob = lib.sdm_observe
    o = [FAKE, FAKE, FAKE, FAKE, 4, 7, 3, 10, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None]
    bad = list(o)
    bad[3] = None                               # class ids missing
    assert ob(*bad) == 1
    bad = list(o)
    bad[7] = 0                                  # no bins
    assert ob(*bad) == 1
    bad = list(o)
    bad[6], bad[5] = 1000, 16                   # counters beyond 48 KB of shared memory
    assert ob(*bad) == 2


def test_threshold_host_validation(lib):
    st = lib.sdm_schedule_threshold
    assert st(None, 4, 7, 0.5, FAKE, FAKE, None, None) == 1
    assert st(FAKE, 0, 7, 0.5, FAKE, FAKE, None, None) == 1
    sw = lib.sdm_threshold_sweep
    assert sw(FAKE, None, 4, 7, None, 3, FAKE, FAKE, FAKE, None, None) == 1      # thresholds missing
    assert sw(FAKE, None, 4, 7, FAKE, 0, FAKE, FAKE, FAKE, None, None) == 1      # K = 0
    assert sw(FAKE, None, 4096, 9, FAKE, 3, FAKE, FAKE, FAKE, None, None) == 2   # R gamma > 32768


def test_binding_checks_the_cost_table():
    import torch
    binding._need_cost(torch.zeros(2 * 4 + 1, dtype=torch.float64), 2, 3)          # R (gamma + 1) + 1 entries
    with pytest.raises(ValueError):
        binding._need_cost(torch.zeros(2 * 4, dtype=torch.float64), 2, 3)          # one short
    with pytest.raises(ValueError):
        binding._need_cost(torch.zeros(2 * 4 + 1, dtype=torch.float32), 2, 3)      # not fp64
