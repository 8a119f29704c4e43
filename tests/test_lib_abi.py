"""The C-ABI library builds, loads and exports every declared symbol (no GPU).

Only host-side paths run here: sizes, status strings and argument
validation, all of which return before any CUDA call.
"""

import ctypes
import os
import re

import pytest

from mixture_experts_layer_91_b300 import binding, build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and nothing else with the moe_ prefix in the dynamic symbol table
    out = os.popen(f"nm -D --defined-only {binding._LIB_PATH}").read()
    exported = sorted(set(re.findall(r"\s(moe_[a-z_0-9]+)$", out, flags=re.M)))
    assert exported == declared_functions()


def test_version_and_status_strings(lib):
    assert lib.moe_version() >> 16 == 2 and lib.moe_version() & 0xffff >= 1
    for s in range(8):
        assert lib.moe_status_string(s).startswith(b"MOE_")
    assert b"unknown" in lib.moe_status_string(99)


def fwd_nulls(lib, c):
    return lib.moe_forward(c, None, None, None, None, None, None, None, None, None, 0,
                           None, None, None, None, None)


def cfg_of(**kw):
    base = dict(T=256, d=128, n_routed=16, n_shared=1, top_k=4, d_ff=64, renormalize=0, gate=0,
                act_dtype=0)
    base.update(kw)
    return binding.MoeConfig(**base)


@pytest.mark.parametrize("bad", [
    dict(top_k=17), dict(top_k=0), dict(d=0), dict(T=-1), dict(n_routed=0), dict(gate=2),
    dict(act_dtype=5), dict(renormalize=2), dict(gate=1, renormalize=0), dict(capacity=-1),
    dict(expert_act=2), dict(combine=2), dict(combine=-1),
])
def test_invalid_configs_rejected(lib, bad):
    c = cfg_of(**bad)
    assert lib.moe_workspace_size(ctypes.byref(c)) == 0
    assert fwd_nulls(lib, ctypes.byref(c)) == 1   # MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(d=12), dict(d_ff=60), dict(n_routed=257),
                                 dict(gate=1, renormalize=1, n_routed=129), dict(top_k=33, n_routed=64)])
def test_unsupported_configs(lib, bad):
    c = cfg_of(**bad)
    st = lib.moe_route(ctypes.byref(c), *([None] * 9), None, 0, None)
    assert st == 2   # MOE_ERR_UNSUPPORTED


def test_null_pointers_and_workspace_checked_before_launch(lib):
    c = cfg_of()
    assert fwd_nulls(lib, None) == 1
    assert lib.moe_route(ctypes.byref(c), *([None] * 9), None, 0, None) == 1
    # a too-small workspace is reported before anything touches the device
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    st = lib.moe_forward(ctypes.byref(c), fake, fake, None, None, None, fake, fake, fake, fake, 16,
                         fake, None, None, None, None)
    assert st == 3   # MOE_ERR_WORKSPACE
    misaligned = ctypes.c_void_p((1 << 20) + 4)
    st = lib.moe_forward(ctypes.byref(c), misaligned, fake, None, None, None, fake, fake, fake, fake,
                         1 << 40, fake, None, None, None, None)
    assert st == 1


@pytest.mark.parametrize("w", workloads.ALL, ids=lambda w: w.name)
def test_workspace_sizes_cover_the_buffers(lib, w):
    c = binding.config(w)
    ws = lib.moe_workspace_size(ctypes.byref(c))
    act = 4 if w.fp32 else 2
    # at least x_perm + H (+ the down projection's bf16 rows, or the fp32
    # accumulator of the scatter-add combine)
    need = act * w.T * w.top_k * w.d + act * (w.n_shared * w.T + w.T * w.top_k) * w.d_ff
    if not w.fp32:
        need += 4 * w.T * w.d if w.combine == "scatter" else 2 * (w.n_shared * w.T + w.T * w.top_k) * w.d
    assert ws >= need
    assert lib.moe_permute_workspace_size(ctypes.byref(c)) >= 4 * w.T * w.top_k
    assert lib.moe_expert_ffn_workspace_size(ctypes.byref(c)) >= act * (w.n_shared * w.T + w.T * w.top_k) * w.d_ff


def test_zero_tokens_is_a_no_op(lib):
    c = cfg_of(T=0)
    assert fwd_nulls(lib, ctypes.byref(c)) == 0
    assert lib.moe_expert_ffn(ctypes.byref(c), None, None, None, None, None, None, None, 0, None,
                              None) == 0
    assert lib.moe_combine(ctypes.byref(c), None, None, None, None, None) == 0


def test_route_workspace_size_matches_the_router_choice(lib):
    """The tensor-core router (bf16, <= 128 router columns, T >= 4096) needs the
    three bf16 planes of [W_g | W_noise] (3 x NP x d x 2 bytes, NP the columns
    rounded up to 32 / 64 / 128) and its fp32 logits rows (T x NP x 4 bytes),
    each region rounded up to 256 bytes. The CUDA-core router needs the split-K
    partial tiles for T <= 512 (token blocks of 32 x 32 splits x 32 tokens x
    EPAD fp32, EPAD the columns rounded up to 32 / 64 / 128 / 256) and one fp32
    logits row of EPAD columns per token above."""
    def up(b):
        return (b + 255) // 256 * 256
    big = dict(T=4096, d=256, act_dtype=1)
    for n_routed, gate, renorm, np_ in [(16, 0, 0, 32), (64, 0, 0, 64), (63, 0, 0, 64), (128, 0, 0, 128),
                                        (16, 1, 1, 32), (64, 1, 1, 128)]:
        c = cfg_of(**big, n_routed=n_routed, gate=gate, renormalize=renorm)
        assert lib.moe_route_workspace_size(ctypes.byref(c)) == up(3 * np_ * 256 * 2) + up(4096 * np_ * 4)
    # CUDA-core router above 512 tokens: one fp32 logits row of EPAD columns per token
    for kw, T, epad in ((dict(T=4095), 4095, 64), (dict(act_dtype=0), 4096, 64), (dict(n_routed=129), 4096, 256),
                        (dict(n_routed=65, gate=1, renormalize=1), 4096, 256)):
        c = cfg_of(**{**big, "n_routed": 64, **kw})
        assert lib.moe_route_workspace_size(ctypes.byref(c)) == T * epad * 4
    for T, n_routed, epad in [(64, 128, 128), (512, 64, 64), (33, 20, 32), (1, 200, 256)]:
        c = cfg_of(**{**big, "T": T, "n_routed": n_routed})
        assert lib.moe_route_workspace_size(ctypes.byref(c)) == (T + 31) // 32 * 32 * 32 * epad * 4
    c = cfg_of(**{**big, "T": 513, "n_routed": 64})
    assert lib.moe_route_workspace_size(ctypes.byref(c)) == 513 * 64 * 4
    # a workspace short of the planes is refused before any launch
    c = cfg_of(**big, n_routed=64)
    fake = ctypes.c_void_p(1 << 20)
    st = lib.moe_route(ctypes.byref(c), fake, fake, None, None, None, fake, fake, None, None, fake, 16, None)
    assert st == 3   # MOE_ERR_WORKSPACE


def test_relu_experts_take_no_w3_but_swiglu_needs_it(lib):
    fake = ctypes.c_void_p(1 << 20)
    for act, want in ((0, 1), (1, 3)):   # SwiGLU: null W3 is an error; ReLU: passes on to the workspace check
        c = cfg_of(expert_act=act, act_dtype=1)
        st = lib.moe_forward(ctypes.byref(c), fake, fake, None, None, None, fake, None, fake, fake, 16,
                             fake, None, None, None, None)
        assert st == want


def test_workspace_follows_the_combine_mode(lib):
    """bf16 layers: MOE_COMBINE_ROWS takes the bf16 rows O [P, d] (P the padded
    H rows), MOE_COMBINE_SCATTER_ADD the fp32 accumulator [T, d]; fp32 layers
    add into y and need neither, whatever the mode."""
    T, d, E, K_s, k, I = 4096, 256, 16, 1, 4, 64
    P = K_s * ((T + 127) // 128) * 128 + T * k + 128 * E
    base = dict(T=T, d=d, n_routed=E, n_shared=K_s, top_k=k, d_ff=I)
    rows = lib.moe_workspace_size(ctypes.byref(cfg_of(**base, act_dtype=1, combine=0)))
    scat = lib.moe_workspace_size(ctypes.byref(cfg_of(**base, act_dtype=1, combine=1)))
    assert rows - scat == 2 * P * d - 4 * T * d
    f0 = lib.moe_workspace_size(ctypes.byref(cfg_of(**base, act_dtype=0, combine=0)))
    f1 = lib.moe_workspace_size(ctypes.byref(cfg_of(**base, act_dtype=0, combine=1)))
    assert f0 == f1 > 0
    assert binding.MOE_COMBINE_ROWS == 0 and binding.MOE_COMBINE_SCATTER_ADD == 1
    assert binding.config(workloads.DSMOE_16B).combine == binding.MOE_COMBINE_ROWS
    assert binding.config(workloads.DSMOE_16B_SCATTER).combine == binding.MOE_COMBINE_SCATTER_ADD


def test_config_struct_matches_the_header():
    """The ctypes mirror of moe_config lists the header's fields in order."""
    src = open(HEADER).read()
    body = src[src.index("typedef struct {\n  int64_t T;"):]
    body = body[:body.index("} moe_config;")]
    names = re.findall(r"\b(?:int64_t|int32_t)\s+(\w+);", body)
    assert names == [f[0] for f in binding.MoeConfig._fields_]


def test_backward_and_training_pair_refuse_bad_arguments_before_any_device_work(lib):
    """moe_backward, moe_backward_from_forward and moe_forward_train check their
    arguments on the host: missing or misaligned pointers give
    MOE_ERR_INVALID_ARG and a workspace below moe_backward_workspace_size()
    MOE_ERR_WORKSPACE, before anything is launched (the fake addresses are never
    dereferenced). moe_forward_train with T = 0 does nothing."""
    c = cfg_of(act_dtype=1, d=256, d_ff=128)
    need = lib.moe_backward_workspace_size(ctypes.byref(c))
    assert need > 0
    f = ctypes.c_void_p(1 << 20)            # 16-byte aligned, never touched
    odd = ctypes.c_void_p((1 << 20) + 2)    # misaligned
    def bwd(fn, *, x=f, dy=f, ws_bytes=need, w1=f, dw1=f, dx=f, extra=()):
        return fn(ctypes.byref(c), x, f, None, None, None, w1, f, f, dy, f, ws_bytes, dx, f, None, dw1, f, f,
                  None, *extra)
    for fn, extra in ((lib.moe_backward, ()), (lib.moe_backward_from_forward, (None,))):
        assert bwd(fn, x=None, extra=extra) == 1
        assert bwd(fn, dy=None, extra=extra) == 1
        assert bwd(fn, w1=None, extra=extra) == 1
        assert bwd(fn, dw1=None, extra=extra) == 1
        assert bwd(fn, dx=odd, extra=extra) == 1
        assert bwd(fn, ws_bytes=need - 1, extra=extra) == 3
    def fwd_train(*, x=f, ws_bytes=need, y=f, T=None):
        cc = c if T is None else cfg_of(act_dtype=1, d=256, d_ff=128, T=T)
        return lib.moe_forward_train(ctypes.byref(cc), x, f, None, None, None, f, f, f, f, ws_bytes, y, None)
    assert fwd_train(x=None) == 1
    assert fwd_train(y=odd) == 1
    assert fwd_train(ws_bytes=need - 1) == 3
    assert fwd_train(T=0, x=None, y=None, ws_bytes=0) == 0
