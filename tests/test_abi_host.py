"""CPU-side checks of the C ABI: the library builds and loads, exports every
function include/kvsel.h declares, and its host-only logic (budget, KV bytes,
argument validation, workspace sizing) agrees with the oracle and the pages.
No compute call is made here (no GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    from query_aware_sparse_block_gb300.build import build_library
    build_library()
    from query_aware_sparse_block_gb300 import kvsel
    kvsel.lib()
    return kvsel


def _declared_functions():
    with open(os.path.join(ROOT, "include", "kvsel.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"KVSEL_API\s+[\w\s\*]+?\b(kvsel_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("kvsel_build_summaries", "kvsel_score_topk", "kvsel_append_score_topk",
              "kvsel_score_topk_window", "kvsel_merge_spans", "kvsel_cache_reset", "kvsel_cache_fetch",
              "kvsel_cache_prefetch", "kvsel_select_scores", "kvsel_selftest_wait_timeout",
              "kvsel_sparse_decode", "kvsel_budget", "kvsel_fetch_spans",
              "kvsel_workspace_size", "kvsel_kv_bytes_per_token", "kvsel_get_error",
              "kvsel_version"):
        assert n in names


def test_library_exports_every_declared_symbol(K):
    L = ctypes.CDLL(K.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(L, n), n
    assert K.kvsel_version().startswith("kvsel")


def test_kv_bytes_per_token_matches_worked_example(K):
    assert K.kvsel_kv_bytes_per_token(32, 2, 128, 2) == 32768
    assert K.kvsel_kv_bytes_per_token(40, 40, 128, 2) == 819200
    assert K.kvsel_kv_bytes_per_token(-1, 2, 128, 2) == -1


def _golden_budget_rows():
    path = os.path.join(ROOT, "tests", "golden", "budget_hand_examples.txt")
    rows = []
    with open(path) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                rows.append(ln.split("|")[0].split())
    return rows


def test_budget_equals_oracle_bit_for_bit(K):
    rows = _golden_budget_rows()
    extra = [["16", "32", "128", "2", "4096", "256", "12e9", "80e12", "2", "0.05", "0.8", "0", "-1"],
             ["64", "2", "128", "2", "4096", "2048", "3.9e11", "1.7376e15", "2", "0.05", "0.8", "0", "-1"],
             ["32", "8", "128", "2", "2560", "1024", "6.7e12", "1.7e15", "2", "0", "1", "1e-7", "0.125"]]
    for r in rows + extra:
        B, H, d, e, hid, N = map(int, r[:6])
        bw, F, kappa, floor, gamma, tau, ovr = map(float, r[6:])
        got = K.kvsel_budget(B, H, d, e, hid, N, bw, F, kappa, floor, gamma, tau, ovr)
        want = o.budget(B, H, d, e, hid, N, bw, F, kappa, floor, gamma, tau, ovr)
        assert got.c_copy_s == want.c_copy_s
        assert got.c_rec_s == want.c_rec_s
        assert got.r_model == want.r_model
        assert got.r == want.r
        assert got.k == want.k
        assert got.tau_rel == want.tau_rel
        assert bool(got.dense) == want.dense


def test_budget_rejects_bad_input(K):
    with pytest.raises(K.KvselError) as ei:
        K.kvsel_budget(64, 2, 128, 2, 4096, 10, 0.0, 1e15)
    assert ei.value.code == K.KVSEL_ERR_INVALID_ARG


def test_workspace_sizes_and_shape_validation(K):
    p = K.problem(16, 32, 8, 128, 32, 1028, 1028)
    assert K.kvsel_workspace_size(p, K.KVSEL_WS_SCORE_TOPK) >= 16 * 1028 * 4
    assert K.kvsel_workspace_size(p, K.KVSEL_WS_SPARSE_DECODE) > 0
    for bad in (K.problem(1, 8, 8, 96, 16, 64), K.problem(1, 8, 3, 64, 16, 64),
                K.problem(1, 64, 2, 128, 16, 64), K.problem(1, 8, 8, 64, 48, 64),
                K.problem(1, 8, 8, 64, 16, 0), K.problem(5000, 8, 8, 64, 16, 64),
                K.problem(1, 8, 8, 64, 16, 64, 65)):
        assert K.kvsel_workspace_size(bad, K.KVSEL_WS_SCORE_TOPK) == 0


def test_entry_points_validate_before_touching_the_device(K):
    bad = K.problem(1, 8, 8, 96, 16, 64)    # head_dim 96 is not compiled
    L = K.lib()
    rc = L.kvsel_score_topk(ctypes.byref(bad), None, None, None, None, 1.0, 0.0, None, None, None,
                            None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_UNSUPPORTED
    good = K.problem(1, 8, 8, 64, 16, 64)
    rc = L.kvsel_score_topk(ctypes.byref(good), None, None, None, None, 1.0, 0.0, None, None, None,
                            None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG
    # the fused append + score call: shape first, then the append inputs, then the rest
    app = K.kvsel_append_in()
    rc = L.kvsel_append_score_topk(ctypes.byref(bad), ctypes.byref(app), None, None, None, 1.0, 0.0,
                                   None, None, None, None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_UNSUPPORTED
    rc = L.kvsel_append_score_topk(ctypes.byref(good), None, None, None, None, 1.0, 0.0, None, None,
                                   None, None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG
    rc = L.kvsel_append_score_topk(ctypes.byref(good), ctypes.byref(app), None, None, None, 1.0, 0.0,
                                   None, None, None, None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG and b"append" in L.kvsel_last_error()
    app.kv_pages, app.n_pages, app.block_table, app.append_pos = 16, 4, 4, 4
    app.summaries, app.open_acc, app.new_v = 16, 16, 16      # new_v without new_k
    rc = L.kvsel_append_score_topk(ctypes.byref(good), ctypes.byref(app), None, None, None, 1.0, 0.0,
                                   None, None, None, None, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG and b"new_v" in L.kvsel_last_error()
    src = K.kvsel_kv_src()
    src.kind = 7
    rc = L.kvsel_sparse_decode(ctypes.byref(good), None, ctypes.byref(src), None, None, None, None,
                               None, None, None, 0.125, None, None, None, None, 0, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG
    rc = L.kvsel_build_summaries(ctypes.byref(good), 9, None, 0, None, None, None, None, None,
                                 None, None, None)
    assert rc == K.KVSEL_ERR_INVALID_ARG
    assert b"mode" in L.kvsel_last_error()


def test_window_entry_point_validates_before_touching_the_device(K):
    L = K.lib()
    good = K.problem(1, 8, 8, 64, 16, 64, 8)
    bad = K.problem(1, 8, 8, 96, 16, 64, 8)

    def call(p, win, app=None):
        return L.kvsel_score_topk_window(ctypes.byref(p), ctypes.byref(win) if win is not None else None,
                                         ctypes.byref(app) if app is not None else None, None, None,
                                         None, None, 1.0, 0.0, None, None, None, None, None, None,
                                         None, None, 0, None)
    assert call(bad, K.kvsel_window(0, 0)) == K.KVSEL_ERR_UNSUPPORTED
    assert call(good, None) == K.KVSEL_ERR_INVALID_ARG
    for n_sink, n_recent in ((-1, 0), (0, -2), (5, 4), (9, 0)):     # k_max = 8
        assert call(good, K.kvsel_window(n_sink, n_recent)) == K.KVSEL_ERR_INVALID_ARG
        assert b"n_sink" in L.kvsel_last_error()
    # a valid window reaches the pointer checks
    assert call(good, K.kvsel_window(4, 4)) == K.KVSEL_ERR_INVALID_ARG
    assert b"NULL pointer" in L.kvsel_last_error()
    app = K.kvsel_append_in()
    assert call(good, K.kvsel_window(1, 1), app) == K.KVSEL_ERR_INVALID_ARG
    assert b"append" in L.kvsel_last_error()


def test_cache_entry_points_validate_before_touching_the_device(K):
    L = K.lib()
    p = K.problem(2, 8, 8, 64, 16, 64, 8)
    assert K.kvsel_workspace_size(p, K.KVSEL_WS_CACHE_FETCH) >= 2 * 9 * 8 + 8
    c = K.kvsel_block_cache()
    assert L.kvsel_cache_reset(ctypes.byref(p), None, None) == K.KVSEL_ERR_INVALID_ARG
    assert L.kvsel_cache_reset(ctypes.byref(p), ctypes.byref(c), None) == K.KVSEL_ERR_INVALID_ARG
    c.pool, c.page_of, c.block_in, c.last_use = 16, 16, 16, 16
    for slots in (7, 4097):                  # below k_max, above the limit
        c.slots = slots
        assert L.kvsel_cache_reset(ctypes.byref(p), ctypes.byref(c), None) == K.KVSEL_ERR_INVALID_ARG
        assert b"slots" in L.kvsel_last_error()
    c.slots = 8

    def fetch(host, step, ws, nws):
        return L.kvsel_cache_fetch(ctypes.byref(p), ctypes.byref(c), host, 64, 4, 4, 4, step, None, 0,
                                   ws, nws, None)
    assert fetch(None, 0, 16, 4096) == K.KVSEL_ERR_INVALID_ARG
    assert fetch(16, -1, 16, 4096) == K.KVSEL_ERR_INVALID_ARG
    assert b"step" in L.kvsel_last_error()
    assert fetch(16, 0, None, 0) == K.KVSEL_ERR_WORKSPACE

    def prefetch(host, pred, ws, nws):
        return L.kvsel_cache_prefetch(ctypes.byref(p), ctypes.byref(c), host, 64, 4, pred, 4, None, 0,
                                      ws, nws, None)
    assert prefetch(None, 4, 16, 4096) == K.KVSEL_ERR_INVALID_ARG
    assert b"cache_prefetch" in L.kvsel_last_error()
    assert prefetch(16, None, 16, 4096) == K.KVSEL_ERR_INVALID_ARG
    assert prefetch(16, 2, 16, 4096) == K.KVSEL_ERR_INVALID_ARG          # misaligned list
    assert b"misaligned" in L.kvsel_last_error()
    assert prefetch(16, 4, None, 0) == K.KVSEL_ERR_WORKSPACE
    c.slots = 7
    assert prefetch(16, 4, 16, 4096) == K.KVSEL_ERR_INVALID_ARG and b"slots" in L.kvsel_last_error()


def test_select_scores_validates_before_touching_the_device(K):
    L = K.lib()
    bad = K.problem(1, 8, 8, 96, 16, 64)

    def call(p, scores=16, gamma=1.0, tau=0.0, k=4):
        return L.kvsel_select_scores(ctypes.byref(p), scores, 4, k, gamma, tau, 4, 4, 4, 4, 4, None,
                                     None)
    assert call(bad) == K.KVSEL_ERR_UNSUPPORTED
    good = K.problem(1, 8, 8, 64, 16, 64)
    assert call(good, scores=None) == K.KVSEL_ERR_INVALID_ARG
    assert call(good, k=None) == K.KVSEL_ERR_INVALID_ARG
    assert call(good, scores=18) == K.KVSEL_ERR_INVALID_ARG and b"misaligned" in L.kvsel_last_error()
    assert call(good, gamma=float("nan")) == K.KVSEL_ERR_INVALID_ARG
    assert call(good, tau=-1.0) == K.KVSEL_ERR_INVALID_ARG
    assert b"tau_rel" in L.kvsel_last_error()
    assert call(K.problem(0, 8, 8, 64, 16, 64)) == K.KVSEL_OK        # empty batch: nothing to do


def test_header_compiles_as_c_and_the_library_links_from_c(K, tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_from_c")
    libdir = os.path.dirname(K.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "abi_from_c.c"), "-L", libdir, "-lkvsel",
           "-Wl,-rpath," + libdir, "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("all ok")


def test_score_path_setting_is_validated(K):
    """kvsel_set_score_path accepts the three forms and returns the previous
    one; an unknown value changes nothing. kvsel_score_path_for names one of
    the two forms (without a GPU: the two-grid form) and rejects a bad shape."""
    L = K.lib()
    assert L.kvsel_set_score_path(7) == -1
    assert K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_TWO_GRID) == K.KVSEL_SCORE_PATH_AUTO
    assert K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_CLUSTER) == K.KVSEL_SCORE_PATH_TWO_GRID
    assert K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_AUTO) == K.KVSEL_SCORE_PATH_CLUSTER
    p = K.problem(16, 32, 8, 128, 32, 1024, 128)
    form, ctas = K.kvsel_score_path_for(p)
    assert form in (K.KVSEL_SCORE_PATH_TWO_GRID, K.KVSEL_SCORE_PATH_CLUSTER)
    assert (ctas == 0) == (form == K.KVSEL_SCORE_PATH_TWO_GRID)
    K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_TWO_GRID)
    assert K.kvsel_score_path_for(p) == (K.KVSEL_SCORE_PATH_TWO_GRID, 0)
    K.kvsel_set_score_path(K.KVSEL_SCORE_PATH_AUTO)
    bad = K.problem(16, 32, 8, 96, 32, 1024, 128)       # head_dim 96 is not supported
    with pytest.raises(K.KvselError):
        K.kvsel_score_path_for(bad)


def test_selftest_divide_validates_arguments(K):
    """kvsel_selftest_divide rejects a negative count of pairs and NULL
    pointers before anything is enqueued; n = 0 is a no-op."""
    import ctypes
    L = K.lib()
    assert L.kvsel_selftest_divide(None, None, None, ctypes.c_int64(-1), None) == K.KVSEL_ERR_INVALID_ARG
    assert L.kvsel_selftest_divide(None, None, None, ctypes.c_int64(0), None) == K.KVSEL_OK
    assert L.kvsel_selftest_divide(None, None, None, ctypes.c_int64(4), None) == K.KVSEL_ERR_INVALID_ARG
