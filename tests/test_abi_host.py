"""CPU-only checks of the C ABI: the library builds, loads, exports every symbol
declared in include/gg.h, and its host-side logic (sizes, buffer carving and
argument validation that rejects before touching the device) behaves as the
header documents. No kernel is launched here."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gg():
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "gg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gg_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for required in ("gg_permute", "gg_grouped_fwd", "gg_swiglu", "gg_grouped_dgrad",
                     "gg_unpermute_combine", "gg_moe_mlp_fwd", "gg_moe_mlp_bwd",
                     "gg_workspace_size", "gg_read_status", "gg_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(gg):
    lib = ctypes.CDLL(gg.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    bound = {n for n, _, _ in gg.SIGNATURES}
    assert set(_declared_functions()) == bound


def test_status_strings_and_version(gg):
    assert gg.version().startswith("gg ")
    for code, name in gg.STATUS_NAMES.items():
        assert gg.status_string(code).startswith(name)
    assert "unknown" in gg.status_string(12345)


def test_workspace_size_grows_with_pairs(gg):
    L = gg.LIB
    assert L.gg_workspace_size(0, 8, 128) >= 256
    assert L.gg_workspace_size(-1, 8, 128) == 0
    # one int32 histogram row of E experts per block of 1024 pairs, at most
    # 128 blocks (larger batches take larger blocks)
    small = L.gg_workspace_size(1000, 8, 128)
    mid = L.gg_workspace_size(16384, 8, 128)
    big = L.gg_workspace_size(131072, 8, 128)
    assert small == 256 + 4 * 128 * 8
    assert mid == big == 256 + 4 * 128 * 128


def _align256(n):
    return (n + 255) // 256 * 256


def _permute_blocks(R):
    """The permute's histogram blocks for R pairs: at most 128 blocks, each a
    whole number of 1024-pair steps (at least one)."""
    per = -(-R // 128)
    ppb = max(1024, -(-per // 1024) * 1024)
    return -(-R // ppb), ppb


def test_workspace_size_matches_the_block_model(gg):
    L = gg.LIB
    for T in (1, 127, 128, 1000, 4096, 16383, 16384, 30272, 131072, 1 << 20):
        for k in (1, 2, 8):
            for E in (1, 8, 128, 1024):
                R = T * k
                nb, ppb = _permute_blocks(R)
                assert 1 <= nb <= 128 and nb * ppb >= R > (nb - 1) * ppb
                assert L.gg_workspace_size(T, k, E) == 256 + _align256(4 * nb * E), (T, k, E)


def test_noalloc_permute_refuses_oversized_batches_on_the_host(gg):
    # The fixed scratch holds 256 KiB of histogram rows: 128 rows of 512
    # experts. Larger batches are refused before any device call, so these
    # never-dereferenced pointers stay untouched.
    L = gg.LIB
    p = ctypes.c_void_p(1 << 40)
    n0 = gg.launch_count()
    # 65544 pairs at E = 1024: 65 rows of 4 KiB
    assert L.gg_permute_noalloc(p, p, p, 8193, 64, 8, 1024, 1, p, p, p, p, p, None) == 4
    assert L.gg_permute_noalloc(p, p, p, 70000, 64, 8, 1024, 1, p, p, p, p, p, None) == 4
    assert L.gg_permute_noalloc(p, p, p, 4096, 64, 8, 1025, 1, p, p, p, p, p, None) == 2
    assert L.gg_permute_noalloc(p, p, p, 4096, 64, 33, 8, 1, p, p, p, p, p, None) == 1
    assert gg.launch_count() == n0


def test_buffers_bind_carves_disjoint_aligned_pieces(gg):
    T, H, F, k, E, P = 300, 320, 384, 2, 8, 16
    n = gg.LIB.gg_moe_buffers_size(T, H, F, k, E, P)
    base = 1 << 40  # never dereferenced: binding is pointer arithmetic only
    buf = gg.GGBuffers()
    assert gg.LIB.gg_moe_buffers_bind(ctypes.c_void_p(base), n, T, H, F, k, E, P,
                                      ctypes.byref(buf)) == 0
    rc = T * k + E * (P - 1)
    sizes = {"Xp": rc * H * 2, "Yp": rc * H * 2, "dYp": rc * H * 2, "dXp": rc * H * 2,
             "H1": rc * 2 * F * 2, "dH": rc * 2 * F * 2, "A": rc * F * 2, "offsets": 4 * (E + 1),
             "row_of_slot": 4 * T * k, "slot_of_row": 4 * rc, "prob_of_row": 4 * rc,
             "rowdot": 4 * rc * gg.LIB.gg_rowdot_stride(F), "ws": buf.ws_bytes}
    spans = sorted((getattr(buf, name), getattr(buf, name) + sz) for name, sz in sizes.items())
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert all(s % 256 == 0 for s, _ in spans)
    assert spans[0][0] >= base and spans[-1][1] <= base + n
    assert buf.ws_bytes >= gg.LIB.gg_workspace_size(T, k, E)
    # too small / misaligned / null
    assert gg.LIB.gg_moe_buffers_bind(ctypes.c_void_p(base), n - 1, T, H, F, k, E, P,
                                      ctypes.byref(buf)) == 4
    assert gg.LIB.gg_moe_buffers_bind(ctypes.c_void_p(base + 16), n, T, H, F, k, E, P,
                                      ctypes.byref(buf)) == 3
    assert gg.LIB.gg_moe_buffers_bind(None, n, T, H, F, k, E, P, ctypes.byref(buf)) == 1


def test_validation_rejects_before_launch(gg):
    L = gg.LIB
    p = ctypes.c_void_p(1 << 40)
    mis = ctypes.c_void_p((1 << 40) + 8)
    ws = ctypes.c_void_p(1 << 41)
    # gg_permute: bad sizes, k > 32, H not a multiple of 64, misaligned x (k > E is
    # legal: a token may name one expert in several slots)
    assert L.gg_permute(p, p, p, 4, 64, 2, 4, 0, p, p, p, p, p, ws, 1 << 20, None) == 1
    assert L.gg_permute(p, p, p, 4, 64, 33, 64, 1, p, p, p, p, p, ws, 1 << 20, None) == 1
    assert L.gg_permute(p, p, p, 4, 96, 2, 4, 1, p, p, p, p, p, ws, 1 << 20, None) == 2
    assert L.gg_permute(p, p, p, 4, 64, 2, 2048, 1, p, p, p, p, p, ws, 1 << 30, None) == 2
    assert L.gg_permute(mis, p, p, 4, 64, 2, 4, 1, p, p, p, p, p, ws, 1 << 20, None) == 3
    assert L.gg_permute(p, p, p, 4, 64, 2, 4, 1, p, p, p, p, p, ws, 16, None) == 4
    assert L.gg_permute(p, None, p, 4, 64, 2, 4, 1, p, p, p, p, p, ws, 1 << 20, None) == 1
    # gg_grouped_fwd: K/N not multiples of 64, wrong epilogue, H1_save or prob with NONE
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 96, 128, 0, p, None, None, ws, 1024, None) == 2
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 100, 0, p, None, None, ws, 1024, None) == 2
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 2, p, None, None, ws, 1024, None) == 1
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 4, p, None, None, ws, 1024, None) == 1
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 5, p, None, None, ws, 1024, None) == 1
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 0, p, p, None, ws, 1024, None) == 1
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 0, p, None, p, ws, 1024, None) == 1
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 192, 1, p, p, None, ws, 1024, None) == 2
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 192, 3, p, p, None, ws, 1024, None) == 2
    assert L.gg_grouped_fwd(mis, p, p, 4, 128, 64, 128, 0, p, None, None, ws, 1024, None) == 3
    assert L.gg_grouped_fwd(p, p, p, 4, 128, 64, 128, 0, p, None, None, ws, 16, None) == 4
    # gg_grouped_dgrad: SwiGLU backward needs H1; NONE must not get H1 or rowdot
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 2, None, None, p, None, ws, 1024,
                              None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 0, p, None, p, None, ws, 1024, None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 0, None, None, p, p, ws, 1024, None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 1, p, None, p, None, ws, 1024, None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 3, p, None, p, None, ws, 1024, None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 4, None, None, p, None, ws, 1024,
                              None) == 1
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 2, p, None, p, mis, ws, 1024, None) == 3
    assert L.gg_grouped_dgrad(p, p, p, 4, 128, 64, 128, 2, p, None, p,
                              ctypes.c_void_p((1 << 40) + 16), ws, 1024, None) == 3
    # gg_unpermute_combine: k > 32, H % 64; dprob needs exactly one of the partial
    # sums or the token-major rows, and neither may come without dprob
    C = L.gg_unpermute_combine
    assert C(p, p, p, 4, 33, 64, 128, p, None, 0, None, None, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 72, 128, p, None, 0, None, None, ws, 1024, None) == 2
    assert C(p, p, p, 4, 2, 64, 128, p, None, 2, None, p, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 64, 128, p, p, 0, None, p, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 64, 128, p, p, 2, None, None, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 64, 128, p, None, 0, p, None, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 64, 128, p, p, 2, p, p, ws, 1024, None) == 1
    assert C(p, p, p, 4, 2, 64, 128, p, None, 0, mis, p, ws, 1024, None) == 3
    assert L.gg_rowdot_blocks(768) == 6 and L.gg_rowdot_blocks(64) == 2
    assert L.gg_rowdot_blocks(256) == 2 and L.gg_rowdot_blocks(0) == 0
    assert L.gg_rowdot_stride(768) == 8 and L.gg_rowdot_stride(1280) == 16
    assert L.gg_rowdot_stride(0) == 0
    # rowdot must be 32-byte aligned
    mis32 = ctypes.c_void_p((1 << 40) + 16)
    assert C(p, p, p, 4, 2, 64, 128, p, mis32, 2, None, p, ws, 1024, None) == 3
    # gg_unpermute_combine_dot: every pointer required, k <= 32, H % 64, alignment
    D = L.gg_unpermute_combine_dot
    assert D(p, p, None, 4, 33, 64, 128, p, p, p, p, ws, 1024, None) == 1
    assert D(p, p, None, 4, 2, 72, 128, p, p, p, p, ws, 1024, None) == 2
    assert D(p, p, None, 4, 2, 64, 128, p, None, p, p, ws, 1024, None) == 1
    assert D(p, p, None, 4, 2, 64, 128, p, p, None, p, ws, 1024, None) == 1
    assert D(p, p, None, 4, 2, 64, 128, p, p, p, None, ws, 1024, None) == 1
    assert D(p, p, None, 4, 2, 64, 128, p, mis, p, p, ws, 1024, None) == 3
    assert D(p, p, None, 4, 2, 64, 128, p, p, mis, p, ws, 1024, None) == 3
    assert D(p, p, None, 4, 2, 64, 128, p, p, p, p, ws, 16, None) == 4
    # gg_ep_split_ids: sizes, El * n_ranks past an int, pointers, workspace
    S = L.gg_ep_split_ids
    assert S(p, -1, 4, 2, p, p, ws, 1024, None) == 1
    assert S(p, 8, 0, 2, p, p, ws, 1024, None) == 1
    assert S(p, 8, 4, 0, p, p, ws, 1024, None) == 1
    assert S(p, 8, 1 << 16, 1 << 16, p, p, ws, 1024, None) == 2
    assert S(None, 8, 4, 2, p, p, ws, 1024, None) == 1
    assert S(p, 8, 4, 2, p, None, ws, 1024, None) == 1
    assert S(p, 8, 4, 2, p, p, ws, 16, None) == 4
    # gg_gather_rows32: sizes, pointers, 4-byte alignment, workspace
    G = L.gg_gather_rows32
    assert G(p, 8, 0, p, 4, p, ws, 1024, None) == 1
    assert G(p, -1, 1, p, 4, p, ws, 1024, None) == 1
    assert G(p, 8, 1, p, -1, p, ws, 1024, None) == 1
    assert G(None, 8, 1, p, 4, p, ws, 1024, None) == 1
    assert G(p, 8, 1, None, 4, p, ws, 1024, None) == 1
    assert G(p, 8, 1, p, 4, None, ws, 1024, None) == 1
    assert G(ctypes.c_void_p((1 << 40) + 2), 8, 1, p, 4, p, ws, 1024, None) == 3
    assert G(p, 8, 1, p, 4, p, ws, 16, None) == 4
    # gg_swiglu / gg_glu: F % 64, only the gated forward epilogues
    assert L.gg_swiglu(p, p, 4, 128, 96, p, None) == 2
    assert L.gg_glu(p, p, 4, 128, 96, 1, None, p, None) == 2
    assert L.gg_glu(p, p, 4, 128, 128, 2, None, p, None) == 1
    assert L.gg_glu(p, p, 4, 128, 128, 0, None, p, None) == 1
    # composites need a full buffer set
    buf = gg.GGBuffers()
    assert L.gg_moe_mlp_fwd(p, p, p, p, p, 4, 64, 128, 2, 4, 1, p, ctypes.byref(buf), None) == 1
    assert L.gg_moe_mlp_bwd(p, p, p, 4, 64, 128, 2, 4, 1, p, None, ctypes.byref(buf), None) == 1
    # options: unknown activation / probability mode; the pre-FC1 backward needs prob
    good = gg.GGBuffers()
    n = L.gg_moe_buffers_size(4, 64, 128, 2, 4, 1)
    assert L.gg_moe_buffers_bind(ctypes.c_void_p(1 << 40), n, 4, 64, 128, 2, 4, 1,
                                 ctypes.byref(good)) == 0
    for act, mode, rec in ((2, 0, 0), (0, 3, 0), (-1, 0, 0), (0, 0, 2)):
        opt = gg.GGOptions(act, mode, rec)
        assert L.gg_moe_mlp_fwd_ex(p, p, p, p, p, 4, 64, 128, 2, 4, 1, ctypes.byref(opt), p,
                                   ctypes.byref(good), None) == 1
        assert L.gg_moe_mlp_bwd_ex(p, p, p, p, p, 4, 64, 128, 2, 4, 1, ctypes.byref(opt), p, p,
                                   ctypes.byref(good), None) == 1
    pre = gg.GGOptions(0, 2, 0)
    assert L.gg_moe_mlp_bwd_ex(p, p, None, p, p, 4, 64, 128, 2, 4, 1, ctypes.byref(pre), p, None,
                               ctypes.byref(good), None) == 1
    assert L.gg_moe_mlp_bwd_ex(p, None, p, p, p, 4, 64, 128, 2, 4, 1, ctypes.byref(pre), p, p,
                               ctypes.byref(good), None) == 1
    assert L.gg_moe_mlp_fwd(p, p, p, p, p, 4, 64, 128, 2, 4, 1, p, None, None) == 1
    assert L.gg_read_status(None, None, None) == 1
    assert L.gg_clear_status(None, None) == 1


def test_mx_layout_and_validation(gg):
    L = gg.LIB
    p = ctypes.c_void_p(1 << 40)
    mis = ctypes.c_void_p((1 << 40) + 8)
    ws = ctypes.c_void_p(1 << 41)
    E, H, F = 4, 256, 384
    lay = gg.mx_weights_layout(E, H, F)
    # four E4M3 operands and their scale tiles, in order, 256-byte aligned, disjoint
    sizes = {"w1": E * 2 * F * H, "w1_scales": E * (F // 128) * (H // 128) * 1024,
             "w2": E * H * F, "w2_scales": E * 1 * (F // 128) * 1024,
             "w2t": E * F * H, "w2t_scales": E * 2 * (H // 128) * 1024,
             "w1t": E * H * 2 * F, "w1t_scales": E * 1 * (2 * F // 128) * 1024}
    spans = sorted((lay[n], lay[n] + sz) for n, sz in sizes.items())
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert all(s % 256 == 0 for s, _ in spans) and spans[-1][1] <= lay["bytes"]
    # shapes: H, F multiples of 128, 0 < E <= 1024
    for bad in ((E, 192, F), (E, H, 320), (0, H, F), (1025, H, F)):
        with pytest.raises(gg.GGError):
            gg.mx_weights_layout(*bad)
    assert L.gg_mx_row_tiles(300, 3, 6, 16) == (300 * 3 + 6 * 15 + 127) // 128 + 6
    assert L.gg_mx_row_tiles(-1, 3, 6, 1) == 0
    # the SwiGLU-backward GEMM runs 128-column tiles, two partials each
    assert L.gg_mx_rowdot_blocks(768) == 12 and L.gg_mx_rowdot_blocks(384) == 6
    assert L.gg_mx_rowdot_blocks(640) == 10 and L.gg_mx_rowdot_stride(640) == 16
    assert L.gg_mx_rowdot_stride(2304) == 40 and L.gg_mx_rowdot_blocks(0) == 0
    # prepare: misaligned buffer, too small
    assert L.gg_mx_prepare_weights(p, p, E, H, F, mis, lay["bytes"], None) == 3
    assert L.gg_mx_prepare_weights(p, p, E, H, F, p, lay["bytes"] - 1, None) == 4
    assert L.gg_mx_prepare_weights(None, p, E, H, F, p, lay["bytes"], None) == 1
    # quantize rows: K % 128, scale capacity, alignment
    R_cap, nt = 900, (900 + 127) // 128 + E
    Q = L.gg_mx_quantize_rows  # T = 300, k = 3, P = 1: R_cap = 900
    assert Q(p, 300, 192, 3, p, p, p, None, E, 1, nt, p, p, p, ws, 1024, None) == 2
    assert Q(p, 300, 256, 3, p, p, p, None, E, 1, nt - 1, p, p, p, ws, 1024, None) == 4
    assert Q(mis, 300, 256, 3, p, p, p, None, E, 1, nt, p, p, p, ws, 1024, None) == 3
    assert Q(p, 300, 256, 33, p, p, p, None, E, 1, nt, p, p, p, ws, 1024, None) == 1
    assert Q(p, 300, 256, 3, None, p, p, None, E, 1, nt, p, p, p, ws, 1024, None) == 1
    assert Q(p, 300, 256, 3, p, p, p, None, E, 0, nt, p, p, p, ws, 1024, None) == 1
    # grouped gemm: outputs each kind needs, activation, capacity, alignment
    G = L.gg_mx_grouped_gemm
    args = (p, p, p, p, E, R_cap, H, F, nt)
    assert G(0, 0, *args, None, None, p, p, None, None, ws, 1024, None) == 1      # FC1 w/o Cq
    assert G(0, 2, *args, None, p, p, p, None, None, ws, 1024, None) == 1         # activation
    assert G(1, 0, *args, None, None, None, None, None, None, ws, 1024, None) == 1  # FC2 w/o C
    assert G(1, 0, *args, p, None, None, None, p, None, ws, 1024, None) == 1      # FC2 + scale
    assert G(2, 0, *args, None, p, p, None, p, None, ws, 1024, None) == 1         # no H1
    assert G(3, 0, *args, p, None, None, None, None, p, ws, 1024, None) == 1      # rowdot
    assert G(4, 0, *args, p, None, None, None, None, None, ws, 1024, None) == 1   # kind
    assert G(1, 0, p, p, p, p, E, R_cap, H, F, nt - 1, p, None, None, None, None, None, ws,
             1024, None) == 4
    assert G(1, 0, mis, p, p, p, E, R_cap, H, F, nt, p, None, None, None, None, None, ws,
             1024, None) == 3
    assert G(2, 0, *args, None, p, p, p, p, ctypes.c_void_p((1 << 40) + 16), ws, 1024,
             None) == 3
    # buffers: disjoint aligned pieces; the layer rejects recompute_h1 and bad shapes
    T, k, P = 300, 3, 16
    n = L.gg_mx_buffers_size(T, H, F, k, E, P)
    buf = gg.GGMxBuffers()
    assert L.gg_mx_buffers_bind(p, n, T, H, F, k, E, P, ctypes.byref(buf)) == 0
    rc = T * k + E * (P - 1)
    ntl = L.gg_mx_row_tiles(T, k, E, P)
    assert buf.n_tiles == ntl
    sizes = {"Xq": rc * H, "Xs": ntl * (H // 128) * 512, "dYq": rc * H,
             "dYs": ntl * (H // 128) * 512, "Aq": rc * F, "As": ntl * (F // 128) * 512,
             "dHq": rc * 2 * F, "dHs": ntl * (2 * F // 128) * 512, "H1": rc * 4 * F,
             "Yp": rc * H * 2, "dXp": rc * H * 2, "offsets": 4 * (E + 1),
             "tiles_before": 4 * (E + 1), "row_of_slot": 4 * T * k, "slot_of_row": 4 * rc,
             "prob_of_row": 4 * rc, "rowdot": 4 * rc * L.gg_mx_rowdot_stride(F),
             "ws": buf.ws_bytes}
    spans = sorted((getattr(buf, name), getattr(buf, name) + sz) for name, sz in sizes.items())
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert all(s % 256 == 0 for s, _ in spans) and spans[-1][1] <= (1 << 40) + n
    assert L.gg_mx_buffers_size(T, 192, F, k, E, P) == 0
    for act, mode, rec in ((0, 0, 1), (2, 0, 0), (0, 3, 0)):
        opt = gg.GGOptions(act, mode, rec)
        assert L.gg_moe_mlp_fwd_mx(p, p, p, p, T, H, F, k, E, P, ctypes.byref(opt), p,
                                   ctypes.byref(buf), None) == 1
        assert L.gg_moe_mlp_bwd_mx(p, p, p, p, T, H, F, k, E, P, ctypes.byref(opt), p, p,
                                   ctypes.byref(buf), None) == 1
    assert L.gg_moe_mlp_fwd_mx(p, p, p, p, T, H, 320, k, E, P, None, p, ctypes.byref(buf),
                               None) == 2
    assert L.gg_moe_mlp_fwd_mx(p, p, p, None, T, H, F, k, E, P, None, p, ctypes.byref(buf),
                               None) == 1
