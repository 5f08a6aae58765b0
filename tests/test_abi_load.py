"""The C-ABI library builds for sm_103a, loads, and exports what include/plmla.h
declares (CPU only: no kernel is launched here)."""
import ctypes

import pytest

import oracle
from paged_latent_attention_gb300 import _native
from paged_latent_attention_gb300.build import build_library


@pytest.fixture(scope="module")
def lib():
    build_library()
    return _native.lib()


def test_every_declared_function_is_exported(lib):
    declared = _native.header_functions()
    assert set(declared) == set(_native.SIGNATURES), "binding table out of sync with header"
    for name in declared:
        assert hasattr(lib, name), name


def test_status_names(lib):
    for code, name in [(0, "PLMLA_OK"), (1, "PLMLA_INVALID_ARGUMENT"), (2, "PLMLA_UNSUPPORTED"),
                       (3, "PLMLA_WORKSPACE_TOO_SMALL"), (4, "PLMLA_CUDA_ERROR")]:
        assert _native.strerror(code) == name
    assert _native.strerror(99) == "PLMLA_UNKNOWN_STATUS"


def _stated_budget(R, n_q, H, slots, min_splits):
    """The library's budget rule as include/plmla.h states it (library tuning
    policy, not part of the method: the pages fix how a budget turns into
    chunks, not the budget itself)."""
    rows = n_q * H
    group = 64 if rows % 64 == 0 else 32 if rows % 32 == 0 else 16
    members = max(1, slots // (rows // group))
    wanted = R * min_splits
    if members > 256 or wanted > 32768:
        return -1
    return min(max(104 * members, wanted), 32768)


@pytest.mark.parametrize("R,n_q,H,slots,min_splits", [
    (64, 1, 64, 152, 1), (32, 1, 64, 152, 1), (128, 4, 64, 152, 1), (4, 1, 64, 152, 128),
    (2, 1, 16, 152, 1), (1, 1, 128, 152, 1), (1000, 2, 48, 148, 3), (7, 3, 16, 16, 2),
    (30, 1, 16, 16, 20), (1, 1, 64, 256, 1), (1024, 1, 64, 152, 8), (1024, 1, 64, 152, 40),
    (1024, 1, 64, 152, 32)])
def test_split_budget_follows_the_stated_rule(lib, R, n_q, H, slots, min_splits):
    assert lib.mla_split_budget(R, n_q, H, slots, min_splits) == _stated_budget(
        R, n_q, H, slots, min_splits)


def test_split_budget_examples(lib):
    # one row group: 104 chunks per persistent CTA on 152 SMs
    assert lib.mla_split_budget(64, 1, 64, 152, 1) == 104 * 152
    # four row groups share the SMs in teams of 38
    assert lib.mla_split_budget(128, 4, 64, 152, 1) == 104 * 38
    # >= 128 chunks for each of 4 million-token requests fits the default budget,
    # and the oracle's planner (pinned by Figure 4) then gives each >= 128 chunks
    b = lib.mla_split_budget(4, 1, 64, 152, 128)
    assert b == 104 * 152
    chunk, splits = oracle.plan_splits([1_000_000] * 4, b, 128)
    assert min(splits) >= 128 and sum(splits) <= b
    # a per-request minimum above the default raises the budget; a larger
    # machine gets a larger one, up to the planner's limit
    assert lib.mla_split_budget(300, 1, 16, 16, 20) == 6000
    assert lib.mla_split_budget(1, 1, 64, 152, 1) > lib.mla_split_budget(1, 1, 64, 16, 1)
    assert lib.mla_split_budget(1, 1, 64, 256, 1) == 104 * 256
    assert lib.mla_split_budget(1024, 1, 64, 152, 32) == 32768
    assert lib.mla_split_budget(1024, 1, 64, 152, 33) == -1


def test_workspace_grows_with_the_machine(lib):
    small = lib.mla_workspace_size(64, 1, 64, 152, 1)
    big = lib.mla_workspace_size(64, 1, 64, 256, 1)
    assert 0 < small < big
    # at most R + members segments of 64 rows x 512 fp32 partials
    assert (64 + 152) * 64 * 512 * 4 <= small < (64 + 152) * 64 * 513 * 4 + (1 << 20)


@pytest.mark.parametrize("args", [(0, 1, 64, 152, 1), (2, 0, 64, 152, 1), (2, 1, 24, 152, 1),
                                  (2, 1, 64, -1, 1), (2, 1, 64, 152, 0), (2000, 1, 64, 152, 1),
                                  (1024, 1, 64, 152, 40)])
def test_bad_shapes_are_rejected_on_the_host(lib, args):
    assert lib.mla_split_budget(*args) == -1
    assert lib.mla_workspace_size(*args) == 0


def test_null_pointers_are_rejected_before_any_launch(lib):
    st = lib.mla_decode(None, None, None, None, 8, 1536 * 576, None, 1, None, 2, 1, 16,
                        ctypes.c_float(0.07), None, None, None, 0, 152, 1, None)
    assert st == 1
    st = lib.mla_split_combine(None, None, None, None, 2, 1, 16, None, None, None)
    assert st == 1
    st = lib.mla_plan_splits(None, 2, 16, None, None, None)
    assert st == 1


def test_misaligned_and_out_of_range_arguments(lib):
    fake = 1 << 20  # never dereferenced: validation fails first
    base = dict(q=fake, qr=fake, g=fake, slab=fake, pages=8, stride=1536 * 576, pt=fake, ld=1,
                lens=fake, R=2, n_q=1, H=16, out=fake, ws=fake)

    def call(**kw):
        a = {**base, **kw}
        return lib.mla_decode(a["q"], a["qr"], a["g"], a["slab"], a["pages"], a["stride"],
                              a["pt"], a["ld"], a["lens"], a["R"], a["n_q"], a["H"],
                              ctypes.c_float(0.07), a["out"], None, a["ws"], 1 << 30, 152, 1,
                              None)
    assert call(q=fake + 2) == 1                 # query not 16-byte aligned
    assert call(stride=1536 * 576 - 8) == 1      # page stride below a page
    assert call(stride=1536 * 576 + 4) == 1      # page stride not a multiple of 8 elements
    assert call(pages=0) == 1
    assert call(H=24) == 1
    assert call(ws=fake + 128) == 1              # workspace not 256-byte aligned


def test_more_than_256_ctas_per_row_group_is_rejected(lib):
    # the persistent schedule keeps per-CTA tables of 256 entries
    assert lib.mla_split_budget(64, 1, 64, 256, 1) > 0
    assert lib.mla_split_budget(64, 1, 64, 257, 1) == -1
    assert lib.mla_workspace_size(64, 1, 64, 257, 1) == 0
    # four row groups: 1024 slots give 256 CTAs per group
    assert lib.mla_split_budget(8, 4, 64, 1024, 1) > 0


def test_query_token_limit_and_fp8_arguments(lib):
    # up to 256 query tokens per request (a chunk of new tokens), not more
    assert lib.mla_split_budget(4, 256, 64, 152, 1) > 0
    assert lib.mla_split_budget(4, 257, 64, 152, 1) == -1
    assert lib.mla_workspace_size_fp8(4, 257, 64, 152, 1) == 0
    # the FP8 workspace adds the two-part queries: 2 x 576 bytes and an exponent per row
    extra = lib.mla_workspace_size_fp8(64, 1, 64, 152, 1) - lib.mla_workspace_size(64, 1, 64, 152, 1)
    assert 64 * 64 * (2 * 576 + 4) <= extra < 64 * 64 * (2 * 576 + 4) + 1024
    fake = 1 << 20

    def fp8(stride=1536 * 576, kv_scale=0.5):
        return lib.mla_decode_fp8(fake, fake, fake, fake, 8, stride, ctypes.c_float(kv_scale), fake,
                                  1, fake, 2, 1, 16, ctypes.c_float(0.07), fake, None, fake, 1 << 30,
                                  152, 1, None)
    assert fp8(stride=1536 * 576 + 8) == 1       # E4M3 page stride not a multiple of 16 bytes
    assert fp8(kv_scale=0.0) == 1
    assert fp8(kv_scale=float("inf")) == 1
    assert fp8(kv_scale=-1.0) == 1
    assert lib.mla_kv_append_fp8(fake, fake, fake, 8, 1536 * 576, ctypes.c_float(0.0), fake, 1,
                                 fake, 1, 1, None, None) == 1
    assert lib.mla_quantize_queries_fp8(fake + 4, fake, 4, fake, fake, None) == 1
    assert lib.mla_quantize_queries_fp8(None, None, 0, None, None, None) == 0


@pytest.mark.parametrize("env,expect", [({}, 0), ({"PLMLA_CHECK_PAGES": "1"}, 1),
                                        ({"PLMLA_DEBUG": "1"}, 1), ({"PLMLA_CHECK_PAGES": "0"}, 0),
                                        ({"PLMLA_DEBUG": ""}, 0)])
def test_page_check_switch_reads_the_environment_at_load(lib, env, expect):
    """Host logic only: the switch's initial value comes from the environment of
    the process that loads the library, and the setter overrides it."""
    import os
    import subprocess
    import sys
    clean = {k: v for k, v in os.environ.items() if k not in ("PLMLA_CHECK_PAGES", "PLMLA_DEBUG")}
    code = ("from paged_latent_attention_gb300 import _native; l = _native.lib(); "
            "a = l.mla_get_page_checks(); l.mla_set_page_checks(1 - a); "
            "print(a, l.mla_get_page_checks())")
    out = subprocess.run([sys.executable, "-c", code], env={**clean, **env}, capture_output=True,
                         text=True, timeout=120, cwd=os.path.dirname(os.path.dirname(__file__)))
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(expect), str(1 - expect)]


@pytest.mark.parametrize("env,expect", [({}, 0), ({"PLMLA_SPLIT_MODE": "uniform"}, 1),
                                        ({"PLMLA_SPLIT_MODE": "per-request"}, 0)])
def test_split_mode_switch(lib, env, expect):
    """Host logic only: the split rule's initial value comes from the
    environment, the setter overrides it, and other modes are rejected."""
    import os
    import subprocess
    import sys
    clean = {k: v for k, v in os.environ.items() if k != "PLMLA_SPLIT_MODE"}
    code = ("from paged_latent_attention_gb300 import _native; l = _native.lib(); "
            "a = l.mla_get_split_mode(); r = l.mla_set_split_mode(1 - a); "
            "bad = l.mla_set_split_mode(2); print(a, l.mla_get_split_mode(), r, bad)")
    out = subprocess.run([sys.executable, "-c", code], env={**clean, **env}, capture_output=True,
                         text=True, timeout=120, cwd=os.path.dirname(os.path.dirname(__file__)))
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(expect), str(1 - expect), "0", "1"]


def test_team_cluster_switch(lib):
    """Host logic only: the widest cluster of query-row teams defaults to 2, the
    setter takes 1, 2 and 4 and rejects anything else."""
    assert lib.mla_get_team_clusters() == 2
    try:
        for v in (1, 4, 2):
            assert lib.mla_set_team_clusters(v) == 0
            assert lib.mla_get_team_clusters() == v
        for bad in (0, 3, 8, -1):
            assert lib.mla_set_team_clusters(bad) == 1
            assert lib.mla_get_team_clusters() == 2
    finally:
        lib.mla_set_team_clusters(2)


def test_layered_decode_arguments_are_checked_on_the_host(lib):
    """mla_decode_layers / _fp8: the layer count, the per-layer pointer arrays
    and the E4M3 scales are validated before any launch."""
    fake = 1 << 20  # never dereferenced: validation fails first
    L = 3
    arr = (ctypes.c_void_p * L)(fake, fake, fake)
    p = ctypes.cast(arr, ctypes.c_void_p)
    holes = (ctypes.c_void_p * L)(fake, None, fake)
    ph = ctypes.cast(holes, ctypes.c_void_p)
    odd = (ctypes.c_void_p * L)(fake, fake + 8, fake)
    po = ctypes.cast(odd, ctypes.c_void_p)

    def call(n=L, q=p, slabs=p, out=p, ws=fake):
        return lib.mla_decode_layers(n, q, p, p, slabs, 8, 1536 * 576, fake, 1, fake, 2, 1, 16,
                                     ctypes.c_float(0.07), out, None, ws, 1 << 30, 152, 1, None)
    assert call(n=0) == 1
    assert call(n=1025) == 1
    assert call(q=None) == 1
    assert call(q=ph) == 1                  # a missing layer pointer
    assert call(out=po) == 1                # a layer's output not 16-byte aligned
    assert call(slabs=ph) == 1
    assert call(ws=fake + 128) == 1
    good = (ctypes.c_float * L)(0.5, 0.25, 1.0)
    bad = (ctypes.c_float * L)(0.5, 0.0, 1.0)

    def call8(scales):
        return lib.mla_decode_layers_fp8(L, p, p, p, p, scales, 8, 1536 * 576, fake, 1, fake, 2,
                                         1, 16, ctypes.c_float(0.07), p, None, fake + 128,
                                         1 << 30, 152, 1, None)
    assert call8(None) == 1
    assert call8(ctypes.cast(bad, ctypes.c_void_p)) == 1
    assert call8(ctypes.cast(good, ctypes.c_void_p)) == 1   # workspace misaligned
