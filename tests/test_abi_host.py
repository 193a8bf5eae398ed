"""The C ABI library on the host, without a GPU: it loads, exports every entry point that
include/gdn.h declares, and rejects bad arguments before any CUDA call.

Only argument errors that the library detects before touching the device are exercised
here; no call in this file reaches a kernel launch.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT

pkg_lib = pytest.importorskip("gated_deltanet_recurrence_03_gb300._lib")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_recurrence_03_gb300 import build
    build.build()
    return pkg_lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and "gdn_recurrent_step" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gdn.h but not exported"
    assert set(names) == set(pkg_lib.EXPORTED)


def test_opts_defaults_and_strings(lib):
    o = pkg_lib.default_opts(lib)
    assert (o.dtype, o.chunk, o.scale, o.flags) == (pkg_lib.GDN_BF16, 64, 1.0, 0)
    assert abs(o.norm_eps - 1e-6) < 1e-12
    assert not o.cu_seqlens and not o.workspace and not o.stream
    assert lib.gdn_status_string(0) == b"ok"
    assert lib.gdn_status_string(pkg_lib.GDN_ERR_TIMEOUT) == b"device-side wait timed out"
    assert lib.gdn_version() >= 300


def opts(lib, **kw):
    o = pkg_lib.default_opts(lib)
    for k, v in kw.items():
        setattr(o, k, v)
    return ctypes.byref(o)


FAKE = 0x10000  # an aligned address that is never dereferenced: every call below fails validation first


def prefill(lib, B=1, T=8, Hqk=1, Hv=1, dk=32, dv=32, ptrs=None, **kw):
    p = [FAKE] * 8 if ptrs is None else ptrs
    return lib.gdn_chunk_fwd(*p, B, T, Hqk, Hv, dk, dv, opts(lib, **kw))


@pytest.mark.parametrize("case,expect", [
    (dict(B=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(T=-5), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(Hqk=2, Hv=3), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(Hqk=0), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(dk=48), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(dv=256), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(chunk=128), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(dtype=7), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(flags=0x80), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(flags=pkg_lib.GDN_RAW_GATES), pkg_lib.GDN_ERR_INVALID_ARG),   # A_log / dt_bias missing
    (dict(flags=pkg_lib.GDN_OUTPUT_GATE), pkg_lib.GDN_ERR_INVALID_ARG),  # z / norm_weight missing
    (dict(ptrs=[FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE + 8] + [FAKE] * 7), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE] * 3 + [FAKE + 1] + [FAKE] * 4), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(B=2, cu_seqlens=FAKE, num_seqs=2), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(cu_seqlens=FAKE, num_seqs=0), pkg_lib.GDN_ERR_INVALID_ARG),
])
def test_prefill_argument_errors(lib, case, expect):
    assert prefill(lib, **case) == expect
    assert lib.gdn_last_error() != b""


@pytest.mark.parametrize("case,expect", [
    (dict(N=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(Hqk=3, Hv=4), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(dk=16), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(null=True), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(misaligned=True), pkg_lib.GDN_ERR_INVALID_ARG),
])
def test_decode_argument_errors(lib, case, expect):
    N, Hqk, Hv, dk, dv = case.get("N", 2), case.get("Hqk", 1), case.get("Hv", 2), case.get("dk", 32), 32
    p = [FAKE] * 7
    if case.get("null"):
        p[5] = 0
    if case.get("misaligned"):
        p[6] = FAKE + 4
    assert lib.gdn_recurrent_step(*p, N, Hqk, Hv, dk, dv, opts(lib)) == expect


def test_empty_calls_do_nothing(lib):
    # no sequences and no tokens: nothing to do, nothing touched
    assert prefill(lib, B=0, T=0, ptrs=[0] * 8) == pkg_lib.GDN_OK
    assert lib.gdn_recurrent_step(*([0] * 7), 0, 1, 1, 32, 32, opts(lib)) == pkg_lib.GDN_OK


def test_workspace_query_is_pure_host(lib):
    # fp32 and small heads take the chunked prefill: per (64-token chunk slot, value head) fp32 T, P
    # (64 x 64), W (64 x dk), U (64 x dv), G (64), the chunk-start state (dk x dv) and the front end's
    # row scalars of k and q (2 x 64); slots = 2 * 8 + 2
    per = 2 * 64 * 64 + 64 * 32 + 64 * 32 + 64 + 32 * 32 + 2 * 64
    need = 18 * 4 * per * 4
    n = lib.gdn_chunk_fwd_workspace_size(2, 512, 4, 4, 32, 32, opts(lib, dtype=pkg_lib.GDN_F32))
    assert need <= n <= need + 7 * 256
    # the in-kernel front end (l2 norm, raw gates) runs inside the same kernels: the same workspace
    for flags in (pkg_lib.GDN_NORMALIZE_QK, pkg_lib.GDN_RAW_GATES, pkg_lib.GDN_NORMALIZE_QK | pkg_lib.GDN_RAW_GATES):
        assert lib.gdn_chunk_fwd_workspace_size(2, 512, 4, 4, 32, 32,
                                                opts(lib, dtype=pkg_lib.GDN_F32, flags=flags)) == n
    assert lib.gdn_chunk_fwd_workspace_size(-1, 512, 4, 4, 32, 32, opts(lib)) == 0


def conv_fwd(lib, B=1, T=8, C=64, K=4, x_stride=0, ptrs=None, **kw):
    p = [FAKE] * 5 if ptrs is None else ptrs   # x, w, cache_in, y, cache_out
    return lib.gdn_causal_conv1d_fwd(p[0], x_stride, p[1], p[2], p[3], p[4], B, T, C, K, opts(lib, **kw))


@pytest.mark.parametrize("case,expect", [
    (dict(C=0), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(C=12), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(K=0), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(K=5), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(B=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(T=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(x_stride=32), pkg_lib.GDN_ERR_INVALID_ARG),                       # narrower than C
    (dict(x_stride=68), pkg_lib.GDN_ERR_INVALID_ARG),                       # bf16 rows lose 16-B alignment
    (dict(dtype=7), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[0] + [FAKE] * 4), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE + 8] + [FAKE] * 4), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE, FAKE, FAKE, FAKE + 4, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(B=2, cu_seqlens=FAKE, num_seqs=2), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(cu_seqlens=FAKE + 2, num_seqs=2), pkg_lib.GDN_ERR_INVALID_ARG),
])
def test_conv_fwd_argument_errors(lib, case, expect):
    assert conv_fwd(lib, **case) == expect
    assert lib.gdn_last_error() != b""


def test_conv_fwd_f32_stride_rule(lib):
    # fp32 rows need a stride that is a multiple of 4 elements; C must still be a multiple of 8
    assert conv_fwd(lib, x_stride=66, dtype=pkg_lib.GDN_F32) == pkg_lib.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, C=20, dtype=pkg_lib.GDN_F32) == pkg_lib.GDN_ERR_INVALID_ARG


@pytest.mark.parametrize("case,expect", [
    (dict(N=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(K=5), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(cache=0), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(y=FAKE + 4), pkg_lib.GDN_ERR_INVALID_ARG),
])
def test_conv_step_argument_errors(lib, case, expect):
    st = lib.gdn_causal_conv1d_step(FAKE, 0, FAKE, case.get("cache", FAKE), case.get("y", FAKE), case.get("N", 4),
                                    64, case.get("K", 4), opts(lib))
    assert st == expect


def test_conv_empty_calls_do_nothing(lib):
    assert conv_fwd(lib, B=0, T=0, ptrs=[0] * 5) == pkg_lib.GDN_OK
    assert lib.gdn_causal_conv1d_step(0, 0, 0, 0, 0, 0, 64, 4, opts(lib)) == pkg_lib.GDN_OK


def conv_qkv(lib, step=False, B=1, T=8, widths=(64, 64, 128), K=4, ptrs=None, **kw):
    p = [FAKE] * 7 if ptrs is None else ptrs   # x, w, cache (in), y_q, y_k, y_v, cache_out
    Cq, Ck, Cv = widths
    if step:
        return lib.gdn_causal_conv1d_step_qkv(p[0], 0, p[1], p[2], p[3], p[4], p[5], B, Cq, Ck, Cv, K, opts(lib, **kw))
    return lib.gdn_causal_conv1d_fwd_qkv(p[0], 0, p[1], p[2], p[3], p[4], p[5], p[6], B, T, Cq, Ck, Cv, K,
                                         opts(lib, **kw))


@pytest.mark.parametrize("step", [False, True])
@pytest.mark.parametrize("case,expect", [
    (dict(widths=(0, 64, 64)), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(widths=(64, 12, 64)), pkg_lib.GDN_ERR_INVALID_ARG),      # not a multiple of 8
    (dict(widths=(64, 64, -8)), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(K=5), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(ptrs=[FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),          # y_k missing
    (dict(ptrs=[FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),   # y_v misaligned
])
def test_conv_qkv_argument_errors(lib, step, case, expect):
    assert conv_qkv(lib, step=step, **case) == expect
    assert lib.gdn_last_error() != b""


def test_conv_qkv_empty_calls_do_nothing(lib):
    assert conv_qkv(lib, B=0, T=0, ptrs=[0] * 7) == pkg_lib.GDN_OK
    assert conv_qkv(lib, step=True, B=0, ptrs=[0] * 7) == pkg_lib.GDN_OK


def bwd(lib, B=1, T=8, Hqk=1, Hv=1, dk=32, dv=32, ptrs=None, **kw):
    p = [FAKE] * 14 if ptrs is None else ptrs
    return lib.gdn_recurrent_bwd(*p, B, T, Hqk, Hv, dk, dv, opts(lib, **kw))


@pytest.mark.parametrize("case,expect", [
    (dict(B=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(Hqk=2, Hv=3), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(dk=48), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(flags=pkg_lib.GDN_NORMALIZE_QK), pkg_lib.GDN_ERR_WORKSPACE),       # front end: validated up to the workspace
    (dict(flags=pkg_lib.GDN_RAW_GATES), pkg_lib.GDN_ERR_INVALID_ARG),        # raw gates need A_log and dt_bias
    (dict(flags=pkg_lib.GDN_RAW_GATES, A_log=FAKE, dt_bias=FAKE, grad_A_log=FAKE + 2), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(flags=pkg_lib.GDN_RAW_GATES, A_log=FAKE, dt_bias=FAKE), pkg_lib.GDN_ERR_WORKSPACE),
    (dict(flags=pkg_lib.GDN_OUTPUT_GATE, z=FAKE, norm_weight=FAKE), pkg_lib.GDN_ERR_UNSUPPORTED),   # no gate backward
    (dict(ptrs=[FAKE] * 8 + [0] + [FAKE] * 5), pkg_lib.GDN_ERR_INVALID_ARG),   # grad_q missing
    (dict(ptrs=[FAKE + 1] + [FAKE] * 13), pkg_lib.GDN_ERR_INVALID_ARG),        # q not element aligned
    (dict(ptrs=[FAKE] * 9 + [FAKE + 2] + [FAKE] * 4), pkg_lib.GDN_ERR_INVALID_ARG),   # grad_k not 4-byte aligned
    (dict(B=2, cu_seqlens=FAKE, num_seqs=2), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(), pkg_lib.GDN_ERR_WORKSPACE),                                      # no workspace
    (dict(workspace=FAKE, workspace_bytes=16), pkg_lib.GDN_ERR_WORKSPACE),    # too small
])
def test_backward_argument_errors(lib, case, expect):
    assert bwd(lib, **case) == expect
    assert lib.gdn_last_error() != b""


def test_backward_optional_pointers_and_empty_calls(lib):
    # S0, grad_S_final and grad_S0 may be NULL; no sequences is a no-op even with no buffers
    assert bwd(lib, B=0, T=0, ptrs=[0] * 14) == pkg_lib.GDN_OK
    p = [FAKE] * 14
    p[5] = p[7] = p[13] = 0
    assert bwd(lib, ptrs=p) == pkg_lib.GDN_ERR_WORKSPACE   # still validated up to the workspace


def test_backward_workspace_size_is_pure_host(lib):
    n = lib.gdn_recurrent_bwd_workspace_size(2, 8192, 16, 32, 128, 128, opts(lib))
    # per (chunk slot, value head), fp32: T, P (64 x 64), W, U, dU (64 x 128), G (64), S, dS (128 x 128);
    # slots = ceil(16384 / 64) + 2 sequences
    per = 2 * 64 * 64 + 3 * 64 * 128 + 64 + 2 * 128 * 128
    need = 258 * 32 * per * 4
    assert need <= n <= need + 8 * 256
    assert lib.gdn_recurrent_bwd_workspace_size(1, 8, 1, 1, 48, 32, opts(lib)) == 0
    # with the front end: the rows' l2 scalars (2 x 64 per slot and value head) join the recurrence's
    # workspace, and fp32 copies of the normalised q, k (tokens x Hqk x dk each), v and dout (tokens x Hv
    # x dv each) and the two gates (tokens x Hv each) follow it
    extra = (258 * 32 * 2 * 64 + 2 * 16384 * 16 * 128 + 2 * 16384 * 32 * 128 + 2 * 16384 * 32) * 4
    for flags in (pkg_lib.GDN_NORMALIZE_QK, pkg_lib.GDN_RAW_GATES, pkg_lib.GDN_NORMALIZE_QK | pkg_lib.GDN_RAW_GATES):
        m = lib.gdn_recurrent_bwd_workspace_size(2, 8192, 16, 32, 128, 128, opts(lib, flags=flags))
        assert n + extra <= m <= n + extra + 8 * 256


@pytest.mark.parametrize("B,T,Hqk,Hv,dk,dv,dtype,nseq", [
    (2, 8192, 16, 32, 128, 128, "bf16", None),    # tensor-core path, batched
    (1, 131072, 16, 32, 128, 128, "bf16", 4),     # tensor-core path, packed
    (3, 97, 2, 6, 128, 128, "bf16", None),        # ragged, odd grouping
    (2, 8192, 16, 32, 128, 128, "f32", None),     # chunked path (fp32)
    (1, 300, 1, 2, 64, 32, "bf16", 5),            # chunked path, packed, small heads
    (4, 512, 4, 4, 32, 32, "bf16", None),         # chunked path, character-LM heads
])
def test_workspace_sizes_follow_the_slot_layout(lib, B, T, Hqk, Hv, dk, dv, dtype, nseq):
    """Both prefill workspaces and the backward workspace, against the slot layout written out here:
    chunk c of sequence i in slot floor(start_i / 64) + i + c, so slots = ceil(tokens / 64) + nseq."""
    packed = nseq is not None
    kw = dict(dtype=pkg_lib.GDN_BF16 if dtype == "bf16" else pkg_lib.GDN_F32)
    if packed:
        kw.update(cu_seqlens=FAKE, num_seqs=nseq)   # the size query only looks at the pointer's presence
    n_seq = nseq if packed else B
    tokens = T if packed else B * T
    slots = -(-tokens // 64) + n_seq
    got = lib.gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, opts(lib, **kw))
    if dtype == "bf16" and dk == dv == 128:
        # per (slot, value head): the 128 x 192 bf16 A1 operand and 128 floats (b_r, gamma_C)
        assert got == slots * Hv * (128 * 192 * 2 + 128 * 4)
    else:
        # fp32 T, P (64 x 64), W (64 x dk), U (64 x dv), G (64), S (dk x dv), row scalars (2 x 64)
        per = 2 * 64 * 64 + 64 * dk + 64 * dv + 64 + dk * dv + 2 * 64
        need = slots * Hv * per * 4
        assert need <= got <= need + 7 * 256
    bwd_kw = dict(kw, dtype=pkg_lib.GDN_BF16 if dtype == "bf16" else pkg_lib.GDN_F32)
    got_b = lib.gdn_recurrent_bwd_workspace_size(B, T, Hqk, Hv, dk, dv, opts(lib, **bwd_kw))
    per_b = 2 * 64 * 64 + 64 * dk + 2 * 64 * dv + 64 + 2 * dk * dv   # + dU (64 x dv) and dS (dk x dv)
    need_b = slots * Hv * per_b * 4
    assert need_b <= got_b <= need_b + 8 * 256


def test_tensor_core_path_accepts_any_head_grouping(lib):
    for Hqk, Hv in ((2, 2), (1, 3), (16, 32)):
        assert lib.gdn_chunk_fwd_workspace_size(1, 512, Hqk, Hv, 128, 128, opts(lib)) > 0


def test_chunk_option_does_not_change_the_path(lib):
    # opts.chunk in {16, 32, 64} is a blocking choice both chunked families serve with 64-token chunks:
    # the same kernels, hence the same workspace, whatever the value (bf16 d=128: the tcgen05 path)
    for dtype, d in ((pkg_lib.GDN_BF16, 128), (pkg_lib.GDN_F32, 32), (pkg_lib.GDN_BF16, 64)):
        sizes = {c: lib.gdn_chunk_fwd_workspace_size(2, 300, 2, 4, d, d, opts(lib, dtype=dtype, chunk=c))
                 for c in (0, 16, 32, 64)}
        assert len(set(sizes.values())) == 1 and sizes[64] > 0, sizes


# ---------------------------------------------------------------- output gate on its own
@pytest.mark.parametrize("case,expect", [
    (dict(rows=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(dv=48), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(dtype=7), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(norm_eps=-1.0), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(ptrs=[FAKE, FAKE, 0, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),         # no norm_weight
    (dict(ptrs=[FAKE, 0, FAKE, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),         # no z
    (dict(ptrs=[FAKE + 8, FAKE, FAKE, FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),  # o not 16-byte aligned
])
def test_output_gate_forward_argument_errors(lib, case, expect):
    p = case.pop("ptrs", [FAKE] * 4)
    rows, dv = case.pop("rows", 8), case.pop("dv", 128)
    assert lib.gdn_output_gate_fwd(*p, rows, dv, opts(lib, **case)) == expect
    assert lib.gdn_last_error() != b""


@pytest.mark.parametrize("case,expect", [
    (dict(rows=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(dv=96), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(ptrs=[FAKE] * 4 + [0] + [FAKE] * 2), pkg_lib.GDN_ERR_INVALID_ARG),          # no grad_o
    (dict(ptrs=[FAKE] * 5 + [FAKE + 4] + [FAKE]), pkg_lib.GDN_ERR_INVALID_ARG),       # grad_z misaligned
    (dict(ptrs=[FAKE] * 6 + [FAKE + 2]), pkg_lib.GDN_ERR_INVALID_ARG),                # grad_norm_weight misaligned
    (dict(), pkg_lib.GDN_ERR_WORKSPACE),                                             # weight sum needs scratch
    (dict(workspace=FAKE, workspace_bytes=64), pkg_lib.GDN_ERR_WORKSPACE),
    (dict(workspace=FAKE + 16, workspace_bytes=1 << 20), pkg_lib.GDN_ERR_INVALID_ARG),   # not 256-byte aligned
])
def test_output_gate_backward_argument_errors(lib, case, expect):
    p = case.pop("ptrs", [FAKE] * 7)
    rows, dv = case.pop("rows", 8), case.pop("dv", 128)
    assert lib.gdn_output_gate_bwd(*p, rows, dv, opts(lib, **case)) == expect
    assert lib.gdn_last_error() != b""


def test_output_gate_sizes_and_empty_calls(lib):
    for dv in (32, 64, 128):   # one partial row of dv floats per block, at most 1024 blocks
        assert lib.gdn_output_gate_bwd_workspace_size(10 ** 6, dv, opts(lib)) == 1024 * dv * 4
    assert lib.gdn_output_gate_bwd_workspace_size(10, 40, opts(lib)) == 0
    assert lib.gdn_output_gate_fwd(0, 0, 0, 0, 0, 128, opts(lib)) == pkg_lib.GDN_OK
    assert lib.gdn_output_gate_bwd(0, 0, 0, 0, 0, 0, 0, 0, 64, opts(lib)) == pkg_lib.GDN_OK   # nothing to write


# ---------------------------------------------------------------- conv backward
def conv_bwd(lib, B=1, T=8, C=64, K=4, ptrs=None, x_stride=0, **kw):
    p = [FAKE] * 8 if ptrs is None else ptrs   # x, w, cache_in, grad_y, grad_cache_out, grad_x, grad_w, grad_cache_in
    return lib.gdn_causal_conv1d_bwd(p[0], x_stride, *p[1:], B, T, C, K, opts(lib, **kw))


@pytest.mark.parametrize("case,expect", [
    (dict(B=-1), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(C=60), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(K=5), pkg_lib.GDN_ERR_UNSUPPORTED),
    (dict(ptrs=[FAKE] * 3 + [0] + [FAKE] * 4), pkg_lib.GDN_ERR_INVALID_ARG),       # no grad_y
    (dict(ptrs=[FAKE] * 5 + [FAKE + 4] + [FAKE] * 2), pkg_lib.GDN_ERR_INVALID_ARG),  # grad_x misaligned
    (dict(B=2, cu_seqlens=FAKE, num_seqs=2), pkg_lib.GDN_ERR_INVALID_ARG),
    (dict(), pkg_lib.GDN_ERR_WORKSPACE),                                           # grad_w needs scratch
])
def test_conv_backward_argument_errors(lib, case, expect):
    assert conv_bwd(lib, **case) == expect
    assert lib.gdn_last_error() != b""


def test_conv_backward_workspace_and_empty(lib):
    # per 64-token slot (ceil(tokens / 64) + sequences of them) one float per channel and tap
    assert lib.gdn_causal_conv1d_bwd_workspace_size(2, 8192, 8192, 4, opts(lib)) == (256 + 2) * 8192 * 4 * 4
    assert lib.gdn_causal_conv1d_bwd_workspace_size(1, 8, 60, 4, opts(lib)) == 0
    assert conv_bwd(lib, B=0, T=0, ptrs=[0] * 8) == pkg_lib.GDN_OK
