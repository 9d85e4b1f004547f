"""Host-only checks of the C ABI: the library loads, exports every entry point
declared in include/la.h, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

import causal_linear_attention_la_gb300 as la
from helpers import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_lib()
    return la.lib()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^LA_API\s+[^(]*?\b(la_\w+)\s*\(", txt, re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared, "no LA_API declarations found"
    assert declared == set(la.exported_symbols)
    for name in declared:
        assert hasattr(lib, name), name
    # and they are real exported symbols of the shared object
    handle = ctypes.CDLL(la.LIBPATH)
    for name in declared:
        getattr(handle, name)


def test_status_strings(lib):
    assert lib.la_status_string(0) == b"LA_OK"
    assert lib.la_status_string(1) == b"LA_ERR_INVALID_ARG"
    assert lib.la_status_string(2) == b"LA_ERR_UNSUPPORTED"
    assert lib.la_status_string(3) == b"LA_ERR_CUDA"
    assert lib.la_status_string(4) == b"LA_ERR_TIMEOUT"
    assert lib.la_status_string(99) == b"LA_ERR_UNKNOWN"
    assert lib.la_version() >= 100


def test_workspace_sizes(lib):
    f = la.la_forward_workspace_size
    assert f(0, 1, 64, 16, 16, 1, la.LA_F32) == 0
    assert f(1, 1, 0, 16, 16, 1, la.LA_F32) == 0
    assert f(1, 1, 64, 48, 16, 1, la.LA_F32) == 0  # unsupported head size
    small = f(1, 1, 64, 16, 16, 1, la.LA_F32)
    assert small >= 4 * (16 * 16 + 16) and small % 256 == 0
    # one record per (b, h, segment); sizes grow with B*H
    assert f(4, 8, 4096, 64, 64, 1, la.LA_BF16) >= 32 * 4 * (64 * 64 + 64)
    b = la.la_backward_workspace_size(4, 8, 8192, 64, 64, 1, la.LA_BF16)
    # state and reverse records (at least one segment each) plus 2 floats per token
    assert b >= 2 * 32 * 4 * (64 * 64 + 64) + 4 * 2 * 32 * 8192
    # the CUDA-core path (fp32 inputs): one state and one reverse record per
    # segment, so the backward needs twice the forward's records plus the tokens
    fs = f(4, 8, 8192, 64, 64, 1, la.LA_F32)
    bs = la.la_backward_workspace_size(4, 8, 8192, 64, 64, 1, la.LA_F32)
    assert bs >= 2 * fs - 256 + 4 * 2 * 32 * 8192


def _fwd(**kw):
    args = dict(q=16, k=32, v=48, out=64, B=1, H=1, N=64, dk=16, dv=16, causal=1,
                eps=1e-6, dtype=la.LA_F32, S_final=None, z_final=None,
                workspace=1024, workspace_bytes=1 << 20, stream=None)
    args.update(kw)
    return la.la_forward(**args)


def test_forward_rejects_bad_arguments(lib):
    # none of these reach the GPU: validation fails first
    assert _fwd(q=None) == la.LA_ERR_INVALID_ARG
    assert b"non-NULL" in lib.la_last_error()
    assert _fwd(k=17) == la.LA_ERR_INVALID_ARG            # misaligned
    assert _fwd(B=-1) == la.LA_ERR_INVALID_ARG
    assert _fwd(dk=24) == la.LA_ERR_UNSUPPORTED
    assert _fwd(dv=256) == la.LA_ERR_UNSUPPORTED
    assert _fwd(dtype=7) == la.LA_ERR_UNSUPPORTED
    assert _fwd(eps=-1.0) == la.LA_ERR_INVALID_ARG
    assert _fwd(eps=float("nan")) == la.LA_ERR_INVALID_ARG
    assert _fwd(eps=float("inf")) == la.LA_ERR_INVALID_ARG
    assert _fwd(workspace=None) == la.LA_ERR_INVALID_ARG
    assert _fwd(workspace_bytes=8) == la.LA_ERR_INVALID_ARG
    assert b"workspace" in lib.la_last_error()
    assert _fwd(S_final=4096) == la.LA_ERR_INVALID_ARG    # z_final missing
    # empty problems are valid and enqueue nothing
    assert _fwd(N=0, q=None, k=None, v=None, out=None) == la.LA_OK
    assert _fwd(B=0) == la.LA_OK
    assert _fwd(H=0, workspace=None, workspace_bytes=0) == la.LA_OK


def test_forward_host_validation(lib):
    """la_forward_host: staging size and argument checks (no GPU reached)."""
    f = la.la_forward_host_workspace_size
    assert f(0, 1, 64, 16, 16, 1, la.LA_F32, 2) == 0
    assert f(1, 1, 64, 24, 16, 1, la.LA_F32, 2) == 0
    # two staging slots of [q | k | v | out] for the largest slice, plus one
    # la_forward workspace for it; more slices, smaller slots
    B, H, N, d = 4, 8, 4096, 64
    one = f(B, H, N, d, d, 1, la.LA_BF16, 1)
    four = f(B, H, N, d, d, 1, la.LA_BF16, 4)
    assert one >= 2 * 4 * B * H * N * d * 2
    assert four >= 2 * 4 * (B * H // 4) * N * d * 2 and four < one
    # slices beyond B*H are clamped: one sequence per slice
    assert f(1, 2, N, d, d, 1, la.LA_BF16, 64) == f(1, 2, N, d, d, 1, la.LA_BF16, 2)
    # ragged slices (B*H not a multiple): slots sized for the larger slice
    assert f(1, 5, N, d, d, 1, la.LA_BF16, 2) >= 2 * 4 * 3 * N * d * 2
    h = dict(q=16, k=32, v=48, out=64, B=1, H=2, N=64, dk=16, dv=16, causal=1, eps=1e-6,
             dtype=la.LA_F32, slices=2, workspace=1024, workspace_bytes=1 << 24, stream=None)
    assert la.la_forward_host(**{**h, "q": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_host(**{**h, "slices": 0}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_host(**{**h, "workspace_bytes": 64}) == la.LA_ERR_INVALID_ARG
    assert b"workspace" in lib.la_last_error()
    assert la.la_forward_host(**{**h, "workspace": 1032}) == la.LA_ERR_INVALID_ARG   # misaligned
    assert la.la_forward_host(**{**h, "dk": 48}) == la.LA_ERR_UNSUPPORTED
    assert la.la_forward_host(**{**h, "eps": -1.0}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_host(**{**h, "N": 0, "q": None}) == la.LA_OK


def test_decode_and_backward_reject_bad_arguments(lib):
    d = dict(S=256, z=512, q=16, k=32, v=48, out=64, B=2, H=2, dk=64, dv=64,
             eps=1e-6, dtype=la.LA_BF16, stream=None)
    assert la.la_decode_step(**{**d, "S": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_step(**{**d, "z": 4}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_step(**{**d, "dk": 96}) == la.LA_ERR_UNSUPPORTED
    assert la.la_decode_step(**{**d, "B": 0}) == la.LA_OK
    b = dict(q=16, k=32, v=48, dout=80, dq=96, dk_=112, dv_=128, B=1, H=1,
             N=64, dk=16, dv=16, causal=1, eps=1e-6, dtype=la.LA_F32,
             workspace=1024, workspace_bytes=1 << 20, stream=None)
    assert la.la_backward(**{**b, "dout": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_backward(**{**b, "workspace_bytes": 4}) == la.LA_ERR_INVALID_ARG
    assert la.la_backward(**{**b, "dv": 8}) == la.LA_ERR_UNSUPPORTED
    assert la.la_backward(**{**b, "N": 0}) == la.LA_OK
    # la_backward_saved: the forward's workspace is required and checked for size
    sv = dict(b, saved=1 << 20, saved_bytes=1 << 20)
    assert la.la_backward_saved(**{**sv, "saved": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_backward_saved(**{**sv, "saved_bytes": 16}) == la.LA_ERR_INVALID_ARG
    assert b"saved" in lib.la_last_error()
    assert la.la_backward_saved(**{**sv, "saved": (1 << 20) + 8}) == la.LA_ERR_INVALID_ARG   # misaligned
    assert la.la_backward_saved(**{**sv, "dv": 8}) == la.LA_ERR_UNSUPPORTED
    assert la.la_backward_saved(**{**sv, "N": 0}) == la.LA_OK


def test_decode_steps_validation(lib):
    """Argument checks of la_decode_steps happen before any device work."""
    d = dict(S=1024, z=1024, q=1024, k=1024, v=1024, out=1024, B=2, H=3, T=4,
             dk=64, dv=64, eps=1e-6, dtype=la.LA_BF16, stream=None)
    assert la.la_decode_steps(**{**d, "T": -1}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps(**{**d, "q": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps(**{**d, "S": 1032}) == la.LA_ERR_INVALID_ARG   # unaligned
    assert la.la_decode_steps(**{**d, "dk": 48}) == la.LA_ERR_UNSUPPORTED
    assert la.la_decode_steps(**{**d, "eps": -1.0}) == la.LA_ERR_INVALID_ARG
    # nothing to do: no device access
    assert la.la_decode_steps(**{**d, "T": 0}) == la.LA_OK
    assert la.la_decode_steps(**{**d, "B": 0}) == la.LA_OK


def test_variant_validation(lib):
    """Argument checks of the variant entry points happen before any device work."""
    d = dict(S=1024, z=1024, q=1024, k=1024, v=1024, out=1024, B=2, H=3, T=4,
             dk=64, dv=64, alpha=2048, eps=1e-6, dtype=la.LA_BF16, stream=None)
    assert la.la_decode_steps_decay(**{**d, "T": -1}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps_decay(**{**d, "alpha": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps_decay(**{**d, "z": 1028}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps_decay(**{**d, "dv": 24}) == la.LA_ERR_UNSUPPORTED
    assert la.la_decode_steps_decay(**{**d, "T": 0}) == la.LA_OK
    e = dict(S=1024, q=1024, k=1024, v=1024, out=1024, B=2, H=3, T=4, dk=64, dv=64,
             dtype=la.LA_F32, stream=None)
    assert la.la_decode_steps_delta(**{**e, "T": -2}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps_delta(**{**e, "k": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_decode_steps_delta(**{**e, "dtype": 7}) == la.LA_ERR_UNSUPPORTED
    assert la.la_decode_steps_delta(**{**e, "H": 0}) == la.LA_OK
    f = dict(q=1024, k=1024, v=1024, out=1024, B=2, H=3, N=100, dk=64, dv=64, alpha=2048, eps=1e-6,
             dtype=la.LA_BF16, S_final=None, z_final=None, workspace=4096, workspace_bytes=1 << 20,
             stream=None)
    assert la.la_forward_decay(**{**f, "dk": 128, "dv": 128}) == la.LA_ERR_UNSUPPORTED
    assert la.la_forward_decay(**{**f, "dtype": la.LA_F32}) == la.LA_ERR_UNSUPPORTED
    assert la.la_forward_decay(**{**f, "alpha": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_decay(**{**f, "S_final": 8192}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_decay(**{**f, "workspace_bytes": 8}) == la.LA_ERR_INVALID_ARG
    assert la.la_forward_decay(**{**f, "N": 0}) == la.LA_OK
    c = dict(dst_S=1024, dst_z=2048, src_S=4096, src_z=8192, B=2, H=3, dk=64, dv=64, stream=None)
    assert la.la_state_copy(**{**c, "dst_z": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_state_copy(**{**c, "src_S": None}) == la.LA_ERR_INVALID_ARG
    assert la.la_state_copy(**{**c, "dst_S": 1030}) == la.LA_ERR_INVALID_ARG
    assert la.la_state_copy(**{**c, "B": 0}) == la.LA_OK


def test_path_selection(lib):
    assert la.la_set_path(42) == -1
    prev = la.la_set_path(la.LA_PATH_SIMT)
    assert la.la_forward_path(64, 64, la.LA_BF16) == 0
    la.la_set_path(la.LA_PATH_AUTO)
    # tensor cores for bf16 with dk = dv in {64, 128}, causal or not
    assert la.la_forward_path(64, 64, la.LA_BF16) == 1
    assert la.la_forward_path(128, 128, la.LA_BF16) == 1
    assert la.la_forward_path(64, 64, la.LA_BF16, False) == 1
    assert la.la_forward_path(128, 128, la.LA_BF16, False) == 1
    assert la.la_forward_path(128, 64, la.LA_BF16) == 0
    assert la.la_forward_path(64, 64, la.LA_F32) == 0
    assert la.la_forward_path(32, 32, la.LA_BF16) == 0
    la.la_set_path(prev)
    assert la.la_forward_path(48, 64, la.LA_BF16) == -1
    assert la.la_forward_path(16, 16, la.LA_F32) == 0


def test_forward_plan_pieces():
    """The causal bf16 forward at d = 128 without a final state takes balanced
    pieces when B*H*P segments would leave SMs idle; with a final state, at
    d = 64, non-causal or fp32 it runs by segments."""
    import causal_linear_attention_la_gb300 as la
    p = la.forward_plan(2, 16, 32768, 128, 128)
    assert (p["pieces"], p["piece_len"]) == (152, 54)
    assert p["pieces"] * p["piece_len"] >= 2 * 16 * 256
    assert la.forward_plan(2, 16, 32768, 128, 128, final_state=True)["pieces"] == 0
    assert la.forward_plan(2, 16, 32768, 128, 128, causal=False)["pieces"] == 0
    assert la.forward_plan(2, 16, 32768, 128, 128, dtype=la.LA_F32)["pieces"] == 0
    assert la.forward_plan(4, 8, 4096, 64, 64)["pieces"] == 0
    # 38 heads of 4 segments already fill the SMs: no pieces
    assert la.forward_plan(2, 19, 27648, 128, 128)["pieces"] == 0
    # the workspace query covers both plans
    ws = la.la_forward_workspace_size(2, 16, 32768, 128, 128, 1, la.LA_BF16)
    assert ws >= 152 * (128 * 128 + 2 * 128) * 4


def test_forward_plan_pieces_invariants():
    """Over many shapes: pieces never exceed one per SM (152), cover every
    chunk of every head, span at most two heads (piece_len <= chunks per head),
    and are taken only where they cost no more than the segment plan, counting
    the records a piece or segment sums (half a chunk each); invalid sizes are
    refused."""
    import causal_linear_attention_la_gb300 as la
    seen = 0
    for BH in (1, 3, 16, 32, 38, 51, 64, 100, 152, 300):
        for N in (100, 640, 1000, 4096, 8192, 32768):
            p = la.forward_plan(1, BH, N, 128, 128)
            nch = -(-N // 128)
            if p["pieces"] == 0:
                continue
            seen += 1
            assert p["pieces"] <= 152
            assert p["pieces"] * p["piece_len"] >= BH * nch > (p["pieces"] - 1) * p["piece_len"]
            assert p["piece_len"] <= nch
            L = -(-p["seg_len"] // 128)
            waves = -(-(BH * p["P"]) // 152)
            ln = p["piece_len"]
            assert (ln + 1) + 0.5 * -(-nch // ln) <= waves * (L + 1) + 0.5 * (p["P"] - 1)
    assert seen > 5
    import ctypes
    buf = (ctypes.c_int * 5)()
    assert la.la_forward_plan(0, 1, 100, 128, 128, 1, la.LA_BF16, 0, ctypes.cast(buf, ctypes.c_void_p)) != la.LA_OK
    assert la.la_forward_plan(1, 1, 100, 48, 128, 1, la.LA_BF16, 0, ctypes.cast(buf, ctypes.c_void_p)) != la.LA_OK
    assert la.la_forward_plan(1, 1, 100, 128, 128, 1, la.LA_BF16, 0, None) != la.LA_OK


def test_forward_plan_few_heads():
    """With few heads the tensor-core plans take fewer, longer segments than
    the CUDA-core plan, since every segment first sums the records of the
    segments before it: one head of 32768 tokens runs in at most 32 segments
    (the CUDA-core plan, which pays no record sums, takes 128), and the chosen
    plan has the lowest modelled cost among all equal-length splits."""
    import causal_linear_attention_la_gb300 as la
    def cost(BH, N, P, L, causal):
        waves = -(-(BH * P) // 152)
        return waves * (L + 1) + 0.02 * P + 0.5 * ((P - 1) if causal else P)
    for BH, N in [(1, 32768), (2, 32768), (4, 32768), (1, 131072), (6, 1000)]:
        for causal in (True, False):
            tc = la.forward_plan(1, BH, N, 128, 128, causal=causal, final_state=True)
            f32 = la.forward_plan(1, BH, N, 128, 128, causal=causal, dtype=la.LA_F32, final_state=True)
            assert tc["P"] <= f32["P"]
            nch = -(-N // 128)
            L = tc["seg_len"] // 128
            best = min(cost(BH, N, P, -(-nch // P), causal) for P in range(1, nch + 1)
                       if -(-nch // -(-nch // P)) == P)
            assert abs(cost(BH, N, tc["P"], L, causal) - best) < 1e-9
    assert la.forward_plan(1, 1, 32768, 128, 128, final_state=True)["P"] <= 32
    assert la.forward_plan(1, 1, 32768, 128, 128, dtype=la.LA_F32, final_state=True)["P"] == 128


def test_backward_workspace_covers_both_plans():
    """The backward's workspace query covers the tensor-core plan (fewer,
    longer segments with few heads) and the CUDA-core plan (more segments):
    two records per (head, segment) of each plus two floats per token."""
    import causal_linear_attention_la_gb300 as la
    rec = (64 * 64 + 64) * 4
    for BH, N in [(1, 32768), (2, 16384), (6, 1000), (32, 8192)]:
        for causal in (1, 0):
            ws = la.la_backward_workspace_size(1, BH, N, 64, 64, causal, la.LA_BF16)
            p_tc = la.forward_plan(1, BH, N, 64, 64, causal=bool(causal), final_state=True)["P"]
            p_cc = la.forward_plan(1, BH, N, 64, 64, causal=bool(causal), dtype=la.LA_F32,
                                   final_state=True)["P"]
            for P in (p_tc, p_cc):
                assert ws >= 2 * BH * P * rec + 8 * BH * N
            assert ws == la.la_backward_workspace_size(1, BH, N, 64, 64, causal, la.LA_F32)
