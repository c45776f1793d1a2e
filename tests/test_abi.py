"""The C-ABI library without a GPU: it loads, exports every function include/fmlp.h declares,
validates arguments before touching any device, and its pure host functions are right."""
import ctypes
import os
import re

import pytest

import feed_forward_gemm_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fmlp.h")

A = 0x10000          # fake, 16-byte aligned "device" addresses; validation never dereferences
GB = 1 << 30


@pytest.fixture(scope="module")
def lib():
    fm.build()
    return fm.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fmlp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("fmlp_linear_bias", "fmlp_mlp_gelu", "fmlp_geglu",
                 "fmlp_geglu_workspace_size", "fmlp_mlp_gelu_workspace_size",
                 "fmlp_status_string", "fmlp_last_error", "fmlp_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fmlp.h but not exported"
    # and the Python binding forwards each under the same name
    for name in declared_functions():
        assert hasattr(fm, name), f"binding lacks {name}"


def test_library_exports_nothing_else(lib):
    out = os.popen(f"nm -D --defined-only {fm.library_path()}").read()
    exported = sorted(set(re.findall(r"\sT\s+(\w+)", out)))
    assert set(exported) == set(declared_functions()), exported


def test_status_strings(lib):
    assert fm.fmlp_status_string(0) == "FMLP_OK"
    for st in range(1, 9):
        assert fm.fmlp_status_string(st).startswith("FMLP_ERR_")
    assert fm.fmlp_version() >= 100


def test_workspace_sizes_and_counts(lib):
    # the [8192, 3072] bf16 intermediate of the GPT-2-small-shaped block: ~50 MB
    assert fm.fmlp_geglu_workspace_size(8192, 768, 3072) == 50_331_648
    assert fm.fmlp_mlp_gelu_workspace_size(4096, 4096, 4096, 4096) in (0, 4096 * 4096 * 2)
    assert fm.fmlp_geglu_workspace_size(0, 768, 3072) == 0


def test_ragged_sizes_plan_as_their_padded_shape(lib):
    """Inner dims that are not multiples of 8 take the plan of the zero-padded shape and need
    no workspace from the caller (the padded path takes its own scratch)."""
    assert fm.fmlp_geglu_plan(8192, 766, 3070) == fm.fmlp_geglu_plan(8192, 768, 3072)
    assert fm.fmlp_mlp_gelu_plan(1, 4093, 4096, 4090) == fm.fmlp_mlp_gelu_plan(1, 4096, 4096, 4096)
    assert fm.fmlp_linear_plan(3, 100, 37) == fm.fmlp_linear_plan(3, 104, 40)
    assert fm.fmlp_geglu_workspace_size(8192, 766, 3072) == 0
    assert fm.fmlp_mlp_gelu_workspace_size(16, 64, 64, 60) == 0
    assert fm.fmlp_geglu_workspace_size(8192, 768, 3072) == 8192 * 3072 * 2


def test_plans_are_pure_host(lib):
    assert fm.fmlp_geglu_plan(0, 768, 3072) == fm.FMLP_PLAN_NONE
    assert fm.fmlp_geglu_plan(8192, 768, 3072) == fm.FMLP_PLAN_TC
    assert fm.fmlp_linear_plan(1024, 32, 64) in (fm.FMLP_PLAN_TC, fm.FMLP_PLAN_GEMV)
    assert fm.fmlp_mlp_gelu_plan(4096, 4096, 4096, 4096) == fm.FMLP_PLAN_TC


def call_linear(x=A, W=A + GB, b=A + 2 * GB, y=A + 3 * GB, T=16, i=32, o=64):
    return fm.fmlp_linear_bias(x, W, b, y, T, i, o, stream=0, raise_on_error=False)


def test_linear_validation(lib):
    assert call_linear(x=0) == fm.FMLP_ERR_NULL
    assert call_linear(W=0) == fm.FMLP_ERR_NULL
    assert call_linear(y=0) == fm.FMLP_ERR_NULL
    assert call_linear(T=-1) == fm.FMLP_ERR_SHAPE
    assert call_linear(i=0) == fm.FMLP_ERR_SHAPE
    # in or out not a multiple of 8: the zero-padded path, with the same checks first
    assert call_linear(i=12, T=0) == fm.FMLP_OK
    assert call_linear(i=12, x=0) == fm.FMLP_ERR_NULL
    assert call_linear(i=12, x=A + 8) == fm.FMLP_ERR_ALIGN
    assert call_linear(o=20, y=A + 16) == fm.FMLP_ERR_ALIAS
    assert call_linear(i=2**31 - 5) == fm.FMLP_ERR_SHAPE
    # ... but a strided call keeps the multiple-of-8 rule
    assert fm.fmlp_linear_bias_strided(A, A + GB, None, A + 3 * GB, 16, 12, 64, ldx=16, ldy=64,
                                       stream=0, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert call_linear(o=2**31) == fm.FMLP_ERR_SHAPE
    assert call_linear(x=A + 8) == fm.FMLP_ERR_ALIGN
    assert call_linear(b=A + 2 * GB + 2) == fm.FMLP_ERR_ALIGN
    assert call_linear(y=A + 16) == fm.FMLP_ERR_ALIAS       # y overlaps x
    assert call_linear(y=A + GB) == fm.FMLP_ERR_ALIAS       # y overlaps W
    assert "overlaps" in fm.fmlp_last_error()
    # T == 0 is a no-op that succeeds without touching pointers or the device
    assert call_linear(T=0, x=0, y=0) == fm.FMLP_OK


def test_transposed_weight_linear_validation(lib):
    def call(**kw):
        a = dict(x=A, Wt=A + GB, b=A + 2 * GB, y=A + 3 * GB, T=16, i=32, o=64)
        a.update(kw)
        return fm.fmlp_linear_bias_wt(a["x"], a["Wt"], a["b"], a["y"], a["T"], a["i"], a["o"],
                                      stream=0, raise_on_error=False)
    assert call(Wt=0) == fm.FMLP_ERR_NULL
    assert call(i=12) == fm.FMLP_ERR_SHAPE            # the TMA row rule: no padded path here
    assert call(Wt=A + GB + 8) == fm.FMLP_ERR_ALIGN
    assert call(y=A + GB + 64) == fm.FMLP_ERR_ALIAS
    assert call(T=0, x=0, y=0) == fm.FMLP_OK


def test_geglu_validation(lib):
    def call(**kw):
        a = dict(x=A, Wg=A + GB, Wu=A + 2 * GB, Wd=A + 3 * GB, y=A + 4 * GB, T=128, D=512,
                 H=128, ws=A + 5 * GB, ws_bytes=128 * 128 * 2)
        a.update(kw)
        return fm.fmlp_geglu(a["x"], a["Wg"], a["Wu"], a["Wd"], a["y"], a["T"], a["D"], a["H"],
                             a["ws"], a["ws_bytes"], stream=0, raise_on_error=False)
    assert call(Wu=0) == fm.FMLP_ERR_NULL
    assert call(H=100, T=0) == fm.FMLP_OK                  # zero-padded path
    assert call(H=100, Wu=0) == fm.FMLP_ERR_NULL
    assert fm.fmlp_geglu_strided(A, A + GB, A + 2 * GB, A + 3 * GB, A + 4 * GB, 128, 512, 100,
                                 A + 5 * GB, 1 << 20, ldx=520, ldy=520, stream=0,
                                 raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert call(ws_bytes=100) == fm.FMLP_ERR_WORKSPACE
    assert call(ws=A + 4 * GB) == fm.FMLP_ERR_ALIAS         # workspace on top of y
    assert call(ws=A + 3 * GB) == fm.FMLP_ERR_ALIAS         # workspace on top of Wd
    assert call(y=A + 2 * GB + 64) == fm.FMLP_ERR_ALIAS
    assert call(Wd=A + 3 * GB + 4) == fm.FMLP_ERR_ALIGN
    assert call(T=0) == fm.FMLP_OK


def test_mlp_validation(lib):
    def call(**kw):
        a = dict(x=A, W1=A + GB, b1=A + 2 * GB, W2=A + 3 * GB, b2=A + 4 * GB, y=A + 5 * GB,
                 T=4, D=64, H=64, Do=64, mode=fm.FMLP_GELU_ERF, ws=A + 6 * GB, ws_bytes=1 << 20)
        a.update(kw)
        return fm.fmlp_mlp_gelu(a["x"], a["W1"], a["b1"], a["W2"], a["b2"], a["y"], a["T"],
                                a["D"], a["H"], a["Do"], a["mode"], a["ws"], a["ws_bytes"],
                                stream=0, raise_on_error=False)
    assert call(W2=0) == fm.FMLP_ERR_NULL
    assert call(mode=7) == fm.FMLP_ERR_SHAPE
    assert call(mode=3, T=0) == fm.FMLP_ERR_SHAPE          # checked before the T == 0 exit
    assert call(mode=fm.FMLP_RELU, T=0) == fm.FMLP_OK
    assert call(Do=6, T=0) == fm.FMLP_OK                   # zero-padded path
    assert call(Do=6, mode=7) == fm.FMLP_ERR_SHAPE
    assert call(Do=6, W2=0) == fm.FMLP_ERR_NULL
    assert call(y=A + 4 * GB) == fm.FMLP_ERR_ALIAS          # y on top of b2
    assert call(T=0) == fm.FMLP_OK


def test_errors_raise_in_python(lib):
    with pytest.raises(fm.FmlpError) as e:
        fm.fmlp_linear_bias(0, A, None, A + GB, 8, 32, 64, stream=0)
    assert e.value.status == fm.FMLP_ERR_NULL and "x is NULL" in str(e.value)


def test_gelu_eval_and_timeout_validation(lib):
    assert fm.fmlp_gelu_eval(A, A + GB, -1, stream=0, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_gelu_eval(A, A + GB, 4, mode=3, stream=0,
                             raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_gelu_eval(0, 0, 0, stream=0, raise_on_error=False) == fm.FMLP_OK
    assert fm.fmlp_gelu_eval(0, 0, 0, mode=fm.FMLP_RELU, stream=0,
                             raise_on_error=False) == fm.FMLP_OK
    assert fm.fmlp_linear_bias_gelu(A, A + GB, None, A + 2 * GB, 8, 32, 64, 3, stream=0,
                                    raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_test_wait_timeout(0, stream=0, raise_on_error=False) == fm.FMLP_ERR_SHAPE


def test_binding_refuses_noncontiguous(lib):
    import torch
    t = torch.zeros(4, 8)[:, ::2]
    with pytest.raises(ValueError):
        fm.fmlp_linear_bias(t, A, None, A + GB, 4, 8, 8, stream=0)


def test_tile_policy_validation(lib):
    assert fm.fmlp_set_tile_policy(7, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    for p in (fm.FMLP_TILES_SINGLE, fm.FMLP_TILES_PAIR, fm.FMLP_TILES_AUTO):
        assert fm.fmlp_set_tile_policy(p) == fm.FMLP_OK


def test_linear_strided_validation_and_view_overlap(lib):
    """Row-strided views: stride rules, and the overlap rule for views of one buffer (exact
    for equal strides, by byte span otherwise). Calls that pass validation stop at the missing
    device here, never at FMLP_ERR_ALIAS."""
    def call(x=A, ldx=1024, y=A + GB, ldy=1024, T=16, i=256, o=512, W=A + 2 * GB, b=None):
        return fm.fmlp_linear_bias_strided(x, W, b, y, T, i, o, ldx=ldx, ldy=ldy, stream=0,
                                           raise_on_error=False)
    assert call(ldx=128) == fm.FMLP_ERR_SHAPE              # ldx < in
    assert call(ldy=256) == fm.FMLP_ERR_SHAPE              # ldy < out
    assert call(ldx=260) == fm.FMLP_ERR_ALIGN              # not a multiple of 8 elements
    assert call(ldy=1028) == fm.FMLP_ERR_ALIGN
    assert call(T=0, x=0, y=0) == fm.FMLP_OK
    # x = buf[:, 0:256], y = buf[:, 256:768] of one [16, 1024] bf16 buffer: disjoint columns
    assert call(x=A, y=A + 256 * 2) not in (fm.FMLP_ERR_ALIAS, fm.FMLP_OK)
    # y = buf[:, 248:760] shares columns 248..255 with x on every row
    assert call(x=A, y=A + 248 * 2) == fm.FMLP_ERR_ALIAS
    assert "overlaps" in fm.fmlp_last_error()
    # y = buf[:, 768:1024] (out = 256) and x = buf[:, 0:256]: disjoint; y starting one row down
    # at columns 0.. of row 1 meets x's row 1
    assert call(x=A, y=A + 768 * 2, o=256) not in (fm.FMLP_ERR_ALIAS, fm.FMLP_OK)
    assert call(x=A, y=A + 1024 * 2, o=256) == fm.FMLP_ERR_ALIAS
    # y entirely below x's last row: no overlap
    assert call(x=A, y=A + 16 * 1024 * 2, o=256) not in (fm.FMLP_ERR_ALIAS, fm.FMLP_OK)
    # different strides whose byte spans meet are treated as overlapping
    assert call(x=A, y=A + 256 * 2, ldy=2048) == fm.FMLP_ERR_ALIAS
    # y may not overlap the packed weight either
    assert call(y=A + 2 * GB + 64) == fm.FMLP_ERR_ALIAS


def test_moe_validation(lib):
    def call(**kw):
        a = dict(x=A, off=A + 6 * GB, E=8, Wg=A + GB, Wu=A + 2 * GB, Wd=A + 3 * GB, y=A + 4 * GB,
                 T=100, D=512, H=1024, ws=A + 5 * GB, ws_bytes=100 * 1024 * 2)
        a.update(kw)
        return fm.fmlp_moe_geglu(a["x"], a["off"], a["Wg"], a["Wu"], a["Wd"], a["y"], a["T"],
                                 a["D"], a["H"], a["E"], a["ws"], a["ws_bytes"], stream=0,
                                 raise_on_error=False)
    assert call(E=0) == fm.FMLP_ERR_SHAPE
    assert call(E=257) == fm.FMLP_ERR_SHAPE
    assert call(D=100) == fm.FMLP_ERR_SHAPE
    assert call(off=0) == fm.FMLP_ERR_NULL
    assert call(off=A + 6 * GB + 2) == fm.FMLP_ERR_ALIGN
    assert call(Wd=A + 3 * GB + 8) == fm.FMLP_ERR_ALIGN
    assert call(ws_bytes=100) == fm.FMLP_ERR_WORKSPACE
    assert call(y=A + 16) == fm.FMLP_ERR_ALIAS              # y on top of x
    assert call(ws=A + 4 * GB) == fm.FMLP_ERR_ALIAS         # workspace on top of y
    assert call(off=A + 4 * GB + 64) == fm.FMLP_ERR_ALIAS   # y on top of the offsets
    assert call(T=0, x=0, y=0) == fm.FMLP_OK
    assert fm.fmlp_moe_geglu_workspace_size(100, 512, 1024) == 100 * 1024 * 2
    assert fm.fmlp_moe_geglu_workspace_size(0, 512, 1024) == 0


def test_decode_crossover_is_pure_host(lib):
    """Blocks of 1..4 tokens take the GEMV pair at one token (and at two for small weights),
    the few-token kernels otherwise (tiny GeGLU blocks the fused one); with the decode switch
    on, the one-kernel decode where it accepts the shape. A single Linear takes the GEMV at
    one token, and at two when its weights are small (<= 16 MiB); the tcgen05 kernels (the
    few-token one below 129 tokens) serve the rest."""
    assert fm.fmlp_mlp_gelu_plan(1, 4096, 4096, 4096) == fm.FMLP_PLAN_GEMV
    assert fm.fmlp_mlp_gelu_plan(4, 4096, 4096, 4096) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(1, 768, 3072) == fm.FMLP_PLAN_GEMV
    assert fm.fmlp_geglu_plan(4, 768, 3072) == fm.FMLP_PLAN_TC
    fm.fmlp_test_prefer_decode(1)
    try:
        assert fm.fmlp_mlp_gelu_plan(1, 4096, 4096, 4096) == fm.FMLP_PLAN_DECODE
        assert fm.fmlp_mlp_gelu_plan(4, 4096, 4096, 4096) == fm.FMLP_PLAN_DECODE
        assert fm.fmlp_geglu_plan(1, 768, 3072) == fm.FMLP_PLAN_DECODE
        assert fm.fmlp_geglu_plan(4, 768, 3072) == fm.FMLP_PLAN_DECODE
        assert fm.fmlp_geglu_plan(1, 8192, 28672) == fm.FMLP_PLAN_GEMV   # no room for two stages
    finally:
        fm.fmlp_test_prefer_decode(0)
    assert fm.fmlp_test_prefer_decode(2, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    # the two-stage switch: -1, 0, 1 accepted; the plan stays FMLP_PLAN_TC either way
    for bad in (2, -2):
        assert fm.fmlp_test_two_stage(bad, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    for mode in (-1, 1, 0):
        assert fm.fmlp_test_two_stage(mode) == fm.FMLP_OK
        assert fm.fmlp_geglu_plan(8192, 768, 3072) == fm.FMLP_PLAN_TC
    assert fm.fmlp_mlp_gelu_plan(5, 4096, 4096, 4096) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(5, 768, 3072) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(1, 32, 64) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_linear_plan(2, 4096, 4096) == fm.FMLP_PLAN_TC       # 33.6 MB
    assert fm.fmlp_linear_plan(2, 256, 64) == fm.FMLP_PLAN_GEMV
    assert fm.fmlp_linear_plan(1, 4104, 520) == fm.FMLP_PLAN_TC        # K not a multiple of 256
    # every plan but the fused one keeps the intermediate in the workspace
    assert fm.fmlp_mlp_gelu_workspace_size(1, 4096, 4096, 4096) == 4096 * 2
    assert fm.fmlp_geglu_workspace_size(3, 768, 3072) == 3 * 3072 * 2
    assert fm.fmlp_geglu_workspace_size(1, 32, 64) == 0


def test_fused_small_plans_are_shape_only(lib):
    """The single-kernel plan of both blocks depends on the shape alone: D (and Dout) up to
    256, H up to 2048; at 1..4 tokens only for tiny weights. Its workspace is 0."""
    assert fm.fmlp_mlp_gelu_plan(1024, 32, 64, 32) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_mlp_gelu_workspace_size(1024, 32, 64, 32) == 0
    assert fm.fmlp_mlp_gelu_plan(100, 40, 72, 48) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_mlp_gelu_plan(100, 40, 72, 40) == fm.FMLP_PLAN_TC         # Dout % 16 != 0
    assert fm.fmlp_mlp_gelu_plan(100, 264, 72, 48) == fm.FMLP_PLAN_TC        # D > 256
    assert fm.fmlp_mlp_gelu_plan(100, 256, 2056, 256) == fm.FMLP_PLAN_TC     # H > 2048
    assert fm.fmlp_mlp_gelu_plan(3, 32, 64, 32) == fm.FMLP_PLAN_FUSED_SMALL  # tiny weights
    assert fm.fmlp_mlp_gelu_plan(3, 256, 2048, 256) == fm.FMLP_PLAN_TC       # 2 MiB of weights
    assert fm.fmlp_mlp_gelu_workspace_size(3, 256, 2048, 256) == 3 * 2048 * 2
    assert fm.fmlp_geglu_plan(3, 256, 2048) == fm.FMLP_PLAN_TC
    assert fm.fmlp_geglu_plan(5, 256, 2048) == fm.FMLP_PLAN_FUSED_SMALL
    assert fm.fmlp_geglu_workspace_size(5, 256, 2048) == 0


def test_injection_hook_validates_its_arguments(lib):
    assert fm.fmlp_test_inject(7, 1, 0, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_test_inject(fm.FMLP_INJECT_LAUNCH, -1, 0, raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_test_inject(fm.FMLP_INJECT_SKIP_LOAD, 1, 3000000,
                               raise_on_error=False) == fm.FMLP_ERR_SHAPE
    assert fm.fmlp_test_inject(fm.FMLP_INJECT_NONE) == fm.FMLP_OK
