"""GPU parity of each kernel against the fp64 oracle, through the C ABI.

Sizes are small enough for the oracle to finish in seconds but span several
128-row tiles, several 256-column tiles, ragged tails in both, an empty expert
and a one-row expert. Index work is compared bit for bit; floating point uses
the parity bar of ``_helpers`` (rel-L2 <= 5e-3, |err| <= 1e-2|ref| + 1e-3)."""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_parity, bits_to_torch, torch_to_bits, torch_to_f64
from moe_synth import normal_bf16

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


@pytest.fixture(scope="module")
def gg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


def _offsets(counts, P=1):
    padded = [-(-c // P) * P for c in counts]
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)


def _nan_filled(shape):
    t = torch.full(shape, 0, dtype=torch.int16, device="cuda")
    t.fill_(NAN_BF16)
    return t.view(torch.bfloat16)


COUNTS = [130, 0, 1, 257, 60]  # ragged, an empty expert, a one-row expert, > 2 row tiles


@pytest.mark.parametrize("K,N", [(320, 320), (64, 256), (192, 576)])
def test_grouped_fwd_plain(gg, K, N):
    rng = np.random.default_rng(K + N)
    E = len(COUNTS)
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 40  # 40 unused rows past offsets[E]
    A = normal_bf16(rng, (R_cap, K), 1.0)
    B = normal_bf16(rng, (E, N, K), 0.05)
    C = _nan_filled((R_cap, N))
    ws = gg.workspace(0, 1, E, "cuda")
    gg.grouped_fwd(bits_to_torch(A), bits_to_torch(B), torch.from_numpy(off).cuda(),
                   gg.GG_EPI_NONE, ws=ws, C=C)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    ref = oracle.grouped_linear(oracle.bf16_bits_to_f64(A), B, off)
    n = int(off[-1])
    assert_parity(torch_to_f64(C[:n]), ref[:n], "C", faithful=oracle.round_to_bf16(ref[:n]))
    # rows past offsets[E] are never written
    assert np.all(torch_to_bits(C[n:]) == NAN_BF16)


@pytest.mark.parametrize("F", [384, 320])
def test_grouped_fwd_swiglu_and_unfused_swiglu(gg, F):
    rng = np.random.default_rng(F)
    E, K = len(COUNTS), 192
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 8
    X = normal_bf16(rng, (R_cap, K), 1.0)
    W1 = normal_bf16(rng, (E, 2 * F, K), 0.08)
    ws = gg.workspace(0, 1, E, "cuda")
    d_off = torch.from_numpy(off).cuda()
    H1 = _nan_filled((R_cap, 2 * F))
    A = _nan_filled((R_cap, F))
    gg.grouped_fwd(bits_to_torch(X), bits_to_torch(W1), d_off, gg.GG_EPI_SWIGLU, ws=ws, C=A,
                   H1_save=H1)
    A2 = _nan_filled((R_cap, F))
    gg.swiglu(H1, d_off, E, A=A2)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    n = int(off[-1])
    h_ref = oracle.grouped_linear(oracle.bf16_bits_to_f64(X), W1, off)
    assert_parity(torch_to_f64(H1[:n]), h_ref[:n], "H1", faithful=oracle.round_to_bf16(h_ref[:n]))
    assert_parity(torch_to_f64(A[:n]), oracle.swiglu(h_ref)[:n], "A",
                  faithful=oracle.round_to_bf16(oracle.swiglu(oracle.round_to_bf16(h_ref)))[:n])
    # fused epilogue and the standalone kernel round alike: bitwise equal
    np.testing.assert_array_equal(torch_to_bits(A[:n]), torch_to_bits(A2[:n]))
    assert np.all(torch_to_bits(A[n:]) == NAN_BF16) and np.all(torch_to_bits(H1[n:]) == NAN_BF16)


@pytest.mark.parametrize("K,N", [(192, 320), (320, 64)])
def test_grouped_dgrad_plain_with_row_scale(gg, K, N):
    rng = np.random.default_rng(7 * K + N)
    E = len(COUNTS)
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 16
    dC = normal_bf16(rng, (R_cap, N), 1.0)
    B = normal_bf16(rng, (E, N, K), 0.05)
    scale = rng.uniform(0.0, 1.0, R_cap).astype(np.float32)
    ws = gg.workspace(0, 1, E, "cuda")
    dA = _nan_filled((R_cap, K))
    gg.grouped_dgrad(bits_to_torch(dC), bits_to_torch(B), torch.from_numpy(off).cuda(),
                     gg.GG_EPI_NONE, prob_of_row=torch.from_numpy(scale).cuda(), ws=ws, dA=dA)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    n = int(off[-1])
    ref = scale.astype(np.float64)[:, None] * oracle.grouped_linear_t(oracle.bf16_bits_to_f64(dC),
                                                                      B, off)
    assert_parity(torch_to_f64(dA[:n]), ref[:n], "dA", faithful=oracle.round_to_bf16(ref[:n]))
    assert np.all(torch_to_bits(dA[n:]) == NAN_BF16)


@pytest.mark.parametrize("F,H", [(320, 256), (256, 128)])
def test_grouped_dgrad_swiglu_backward(gg, F, H):
    rng = np.random.default_rng(F * 3 + H)
    E = len(COUNTS)
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 16
    dY = normal_bf16(rng, (R_cap, H), 1.0)
    W2 = normal_bf16(rng, (E, H, F), 0.05)
    H1 = normal_bf16(rng, (R_cap, 2 * F), 1.5)
    prob = rng.uniform(0.05, 1.0, R_cap).astype(np.float32)
    ws = gg.workspace(0, 1, E, "cuda")
    dH = _nan_filled((R_cap, 2 * F))
    nb, nbs = gg.rowdot_blocks(F), gg.rowdot_stride(F)
    rowdot = torch.full((R_cap, nbs), float("nan"), dtype=torch.float32, device="cuda")
    gg.grouped_dgrad(bits_to_torch(dY), bits_to_torch(W2), torch.from_numpy(off).cuda(),
                     gg.GG_EPI_SWIGLU_BWD, H1=bits_to_torch(H1),
                     prob_of_row=torch.from_numpy(prob).cuda(), ws=ws, dA=dH, rowdot=rowdot)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    n = int(off[-1])
    acc = oracle.grouped_linear_t(oracle.bf16_bits_to_f64(dY), W2, off)
    dA = prob.astype(np.float64)[:, None] * acc
    h1 = oracle.bf16_bits_to_f64(H1)
    ref = oracle.swiglu_backward(dA, h1)
    assert_parity(torch_to_f64(dH[:n]), ref[:n], "dH", faithful=oracle.round_to_bf16(ref[:n]))
    assert np.all(torch_to_bits(dH[n:]) == NAN_BF16)
    # dprob partial sums: block b = columns [128 b, 128 b + 128) of the unscaled
    # accumulator against the forward's BF16 SwiGLU output
    a = oracle.round_to_bf16(oracle.swiglu(h1))
    prod = acc * a
    ref_rd = np.stack([prod[:, 128 * b:128 * (b + 1)].sum(axis=1) for b in range(nb)], axis=1)
    got_rd = rowdot.cpu().numpy().astype(np.float64)
    assert_parity(got_rd[:n, :nb], ref_rd[:n], "rowdot")
    assert np.all(np.isnan(got_rd[n:]))  # rows past offsets[E] are not written
    assert np.all(np.isnan(got_rd[:, nb:]))  # nor the padding of each row's group


def _permute_case(T, E, k, seed, skew=None, dup=False):
    rng = np.random.default_rng(seed)
    if dup:
        idx = rng.integers(0, E, size=(T, k))
    elif skew is not None:
        idx = np.full((T, k), skew)
        if k > 1:
            idx[:, 1:] = (skew + 1 + np.arange(k - 1)) % E
    else:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]) if T else \
            np.zeros((0, k), np.int64)
    prob = rng.uniform(0, 1, (T, k)).astype(np.float32)
    return idx.astype(np.int32).reshape(T, k), prob


@pytest.mark.parametrize("T,H,E,k,P,extra", [
    (256, 64, 4, 2, 1, {}), (300, 256, 8, 2, 1, {}), (300, 256, 8, 2, 16, {}),
    (1, 64, 1, 1, 1, {}), (5000, 128, 16, 1, 1, {"skew": 7}), (3000, 64, 1024, 8, 1, {}),
    (700, 192, 6, 3, 256, {"dup": True}), (4096, 64, 128, 8, 256, {}),
    # more slots than experts (the grouping by rank of expert parallelism)
    (600, 64, 2, 8, 1, {"dup": True}), (300, 128, 4, 8, 16, {"dup": True}),
    # rows of several 1 KB slices for the padding zeroing (H = 1344: 64 + 64 + 40
    # vectors), long runs of padding rows (P = 256)
    (512, 2048, 16, 4, 256, {}), (300, 1344, 8, 2, 64, {"skew": 3}),
])
def test_permute_bit_exact(gg, T, H, E, k, P, extra):
    idx, prob = _permute_case(T, E, k, T + E, **extra)
    x = normal_bf16(np.random.default_rng(1), (T, H), 1.0)
    # NaN where nothing is written: a padding row left unzeroed fails below
    Xp = torch.full((gg.r_cap(T, k, E, P), H), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = gg.permute(bits_to_torch(x), torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(),
                     E, P, out={"Xp": Xp})
    torch.cuda.synchronize()
    assert gg.read_status(out["ws"]) == 0
    off, ros, sor = oracle.route(idx, E, P)
    np.testing.assert_array_equal(out["offsets"].cpu().numpy(), off)
    np.testing.assert_array_equal(out["row_of_slot"].cpu().numpy(), ros)
    np.testing.assert_array_equal(out["slot_of_row"].cpu().numpy(), sor)
    por = out["prob_of_row"].cpu().numpy()
    live = sor >= 0
    np.testing.assert_array_equal(por[live], prob.reshape(-1)[sor[live]])
    assert np.all(por[~live] == 0)
    n = int(off[-1])
    xp = torch_to_bits(out["Xp"][:n])
    live_n = sor[:n] >= 0
    np.testing.assert_array_equal(xp[live_n], x[sor[:n][live_n] // k])
    assert np.all(xp[~live_n] == 0)


def test_permute_empty_batch_writes_zero_offsets(gg):
    E = 8
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    prob = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    out = gg.permute(x, idx, prob, E, 4, out={"offsets": torch.full((E + 1,), 7, dtype=torch.int32,
                                                                     device="cuda")})
    torch.cuda.synchronize()
    assert np.all(out["offsets"].cpu().numpy() == 0)


@pytest.mark.parametrize("weighted", [True, False])
def test_combine(gg, weighted):
    T, H, E, k = 333, 192, 8, 3
    idx, prob = _permute_case(T, E, k, 5)
    x = normal_bf16(np.random.default_rng(2), (T, H), 1.0)
    p = gg.permute(bits_to_torch(x), torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(), E, 4)
    R_cap = p["Xp"].shape[0]
    Yp = normal_bf16(np.random.default_rng(3), (R_cap, H), 1.0)
    out = gg.unpermute_combine(bits_to_torch(Yp), p["row_of_slot"],
                               torch.from_numpy(prob).cuda() if weighted else None, T, k, p["ws"])
    torch.cuda.synchronize()
    assert gg.read_status(p["ws"]) == 0
    ros = p["row_of_slot"].cpu().numpy()
    ref = oracle.combine(oracle.bf16_bits_to_f64(Yp), ros, prob if weighted else None, T, k)
    assert_parity(torch_to_f64(out), ref, "out", faithful=oracle.round_to_bf16(ref))


def test_combine_prob_gradient_sums_partials_in_order(gg):
    # dprob[t, j] = sum_b rowdot[b][row(t, j)] in fp32, b ascending: bit-exact
    # against the same fp32 sum on the host; a pair without a row gives 0.
    T, k, H, R_cap = 300, 3, 64, 1000
    rng = np.random.default_rng(41)
    rows = rng.permutation(R_cap)[:T * k].astype(np.int32)
    rows[[5, 77, 301]] = -1
    Yp = normal_bf16(rng, (R_cap, H), 1.0)
    ws = gg.workspace(T, k, 1, "cuda")
    # one group of 8 with padding, exactly one, two groups (padded, exact),
    # and partials past the 16 loaded before the column loop
    for nb in (6, 8, 11, 16, 19):
        nbs = (nb + 7) // 8 * 8
        rowdot = np.full((R_cap, nbs), np.nan, np.float32)
        rowdot[:, :nb] = rng.standard_normal((R_cap, nb))
        out, dprob = gg.unpermute_combine(bits_to_torch(Yp), torch.from_numpy(rows).cuda(), None,
                                          T, k, ws, rowdot=torch.from_numpy(rowdot).cuda(),
                                          n_rowdot=nb)
        torch.cuda.synchronize()
        assert gg.read_status(ws) == 0
        want = np.zeros(T * k, np.float32)
        for b in range(nb):
            want = np.where(rows >= 0, want + rowdot[np.maximum(rows, 0), b], want)
            want = want.astype(np.float32)
        np.testing.assert_array_equal(dprob.cpu().numpy().reshape(-1), want)
    # the combine itself is unchanged by the extra output
    out2 = gg.unpermute_combine(bits_to_torch(Yp), torch.from_numpy(rows).cuda(), None, T, k, ws)
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out2))


@pytest.mark.parametrize("T,H,E,k,P", [(400, 128, 8, 2, 8), (257, 1344, 6, 3, 128)])
def test_permute_rows_gathers_token_gradient(gg, T, H, E, k, P):
    idx, prob = _permute_case(T, E, k, 9)
    x = normal_bf16(np.random.default_rng(4), (T, H), 1.0)
    dO = normal_bf16(np.random.default_rng(5), (T, H), 1.0)
    p = gg.permute(bits_to_torch(x), torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(), E, P)
    R_cap = p["Xp"].shape[0]
    dst = torch.full((R_cap, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dYp = gg.permute_rows(bits_to_torch(dO), p["row_of_slot"], p["slot_of_row"], p["offsets"], k,
                          E, P, R_cap, p["ws"], dst=dst)
    torch.cuda.synchronize()
    sor = p["slot_of_row"].cpu().numpy()
    n = int(p["offsets"][-1].item())
    got = torch_to_bits(dYp[:n])
    live = sor[:n] >= 0
    np.testing.assert_array_equal(got[live], dO[sor[:n][live] // k])
    assert np.all(got[~live] == 0)


def test_ep_split_ids(gg):
    # owning rank and local expert of every pair; an id outside [0, El * W)
    # gives -1 for both and the bad-expert status
    El, W, T, k = 6, 4, 300, 3
    rng = np.random.default_rng(21)
    idx = rng.integers(0, El * W, size=(T, k)).astype(np.int32)
    idx[7, 1] = El * W
    idx[9, 0] = -2
    ws = gg.workspace(T, k, W, "cuda")
    dest, leid = gg.ep_split_ids(torch.from_numpy(idx).cuda(), El, W, ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 16
    ok = (idx >= 0) & (idx < El * W)
    np.testing.assert_array_equal(dest.cpu().numpy(), np.where(ok, idx // El, -1))
    np.testing.assert_array_equal(leid.cpu().numpy(), np.where(ok, idx % El, -1))


@pytest.mark.parametrize("width", [1, 3])
def test_gather_rows32(gg, width):
    rng = np.random.default_rng(22 + width)
    R, n = 57, 400
    src = rng.standard_normal((R, width)).astype(np.float32)
    index = rng.integers(-1, R, size=n).astype(np.int32)
    ws = gg.workspace(1, 1, 1, "cuda")
    s_t = torch.from_numpy(src if width > 1 else src[:, 0].copy()).cuda()
    got = gg.gather_rows32(s_t, torch.from_numpy(index).cuda(), ws).cpu().numpy()
    ref = np.where((index >= 0)[:, None], src[np.maximum(index, 0)], 0.0)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    np.testing.assert_array_equal(got.reshape(n, width), ref)  # bit-exact copies
    # int32 rows travel unchanged too; an index past the rows zeroes and flags
    index[5] = R
    got_i = gg.gather_rows32(torch.arange(R * width, dtype=torch.int32).reshape(
        (R, width) if width > 1 else (R,)).cuda(), torch.from_numpy(index).cuda(), ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 18
    gi = got_i.cpu().numpy().reshape(n, width)
    live = (index >= 0) & (index < R)
    np.testing.assert_array_equal(gi[live], (index[live, None] * width + np.arange(width)))
    assert np.all(gi[~live] == 0)


def test_device_status_bad_expert_id(gg):
    T, H, E, k = 64, 64, 4, 2
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[5, 1] = 9   # out of range
    idx[6, 0] = -2  # out of range
    prob = np.ones((T, k), np.float32)
    x = normal_bf16(np.random.default_rng(0), (T, H), 1.0)
    p = gg.permute(bits_to_torch(x), torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(), E, 1)
    torch.cuda.synchronize()
    assert gg.read_status(p["ws"]) == 16
    ros = p["row_of_slot"].cpu().numpy()
    assert ros[5 * k + 1] == -1 and ros[6 * k] == -1
    assert int(p["offsets"][-1].item()) == T * k - 2
    gg.clear_status(p["ws"])
    assert gg.read_status(p["ws"]) == 0


def test_device_status_bad_offsets_computes_nothing(gg):
    E, K, N, R_cap = 3, 64, 64, 256
    A = torch.zeros((R_cap, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((E, N, K), dtype=torch.bfloat16, device="cuda")
    C = _nan_filled((R_cap, N))
    ws = gg.workspace(0, 1, E, "cuda")
    bad = torch.tensor([0, 100, 50, 200], dtype=torch.int32, device="cuda")  # not monotone
    gg.grouped_fwd(A, B, bad, gg.GG_EPI_NONE, ws=ws, C=C)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 17
    assert np.all(torch_to_bits(C) == NAN_BF16)
    gg.clear_status(ws)
    too_far = torch.tensor([0, 100, 200, 300], dtype=torch.int32, device="cuda")  # > R_cap
    gg.grouped_fwd(A, B, too_far, gg.GG_EPI_NONE, ws=ws, C=C)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 17


def test_bounded_wait_times_out_and_context_survives(gg):
    ws = gg.workspace(0, 1, 1, "cuda")
    gg.selftest_bounded_wait(ws, 2_000_000)  # 2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 19
    # the context is still usable afterwards
    gg.clear_status(ws)
    test_grouped_fwd_plain(gg, 64, 256)


@pytest.mark.parametrize("P,T,E,k,H,F", [(1, 300, 8, 2, 256, 320), (16, 257, 6, 3, 320, 384),
                                         (256, 700, 5, 2, 192, 256)])
def test_gathered_gemms_equal_materialised_path(gg, P, T, E, k, H, F):
    # FC1 on the gathered x rows == FC1 on gg_permute's Xp; dgrad FC2 on the
    # gathered dOut rows == dgrad FC2 on gg_permute_rows' dYp: bit for bit,
    # including zero padding rows and the rows of empty experts.
    idx, prob = _permute_case(T, E, k, 17 + P)
    idx[idx == 1] = 0  # expert 1 gets no tokens
    rng = np.random.default_rng(P + T)
    x = bits_to_torch(normal_bf16(rng, (T, H), 1.0))
    dO = bits_to_torch(normal_bf16(rng, (T, H), 1.0))
    W1 = bits_to_torch(normal_bf16(rng, (E, 2 * F, H), 0.05))
    W2 = bits_to_torch(normal_bf16(rng, (E, H, F), 0.05))
    p = gg.permute(x, torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(), E, P)
    R_cap = p["Xp"].shape[0]
    n = int(p["offsets"][-1].item())
    ws = p["ws"]
    for epi in (gg.GG_EPI_SWIGLU, gg.GG_EPI_QGEGLU, gg.GG_EPI_NONE):
        gated = epi != gg.GG_EPI_NONE
        H1a = _nan_filled((R_cap, 2 * F)) if gated else None
        H1b = _nan_filled((R_cap, 2 * F)) if gated else None
        ncols = F if gated else 2 * F
        Ca, Cb = _nan_filled((R_cap, ncols)), _nan_filled((R_cap, ncols))
        gg.grouped_fwd(p["Xp"], W1, p["offsets"], epi, ws=ws, C=Ca, H1_save=H1a)
        gg.grouped_fwd_gather(x, p["slot_of_row"], k, W1, p["offsets"], epi, ws=ws, C=Cb,
                              H1_save=H1b)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(torch_to_bits(Ca), torch_to_bits(Cb))
        if H1a is not None:
            np.testing.assert_array_equal(torch_to_bits(H1a), torch_to_bits(H1b))
    H1 = bits_to_torch(normal_bf16(rng, (R_cap, 2 * F), 1.0))
    dYp = gg.permute_rows(dO, p["row_of_slot"], p["slot_of_row"], p["offsets"], k, E, P, R_cap, ws)
    for epi in (gg.GG_EPI_SWIGLU_BWD, gg.GG_EPI_QGEGLU_BWD, gg.GG_EPI_NONE):
        # dgrad through W2 [E][H][F]: [R][2F] with a gated backward, else [R][F]
        gated = epi != gg.GG_EPI_NONE
        ncols = 2 * F if gated else F
        da, db = _nan_filled((R_cap, ncols)), _nan_filled((R_cap, ncols))
        h1 = H1 if gated else None
        gg.grouped_dgrad(dYp, W2, p["offsets"], epi, H1=h1, prob_of_row=p["prob_of_row"], ws=ws,
                         dA=da)
        gg.grouped_dgrad_gather(dO, p["slot_of_row"], k, W2, p["offsets"], epi, H1=h1,
                                prob_of_row=p["prob_of_row"], ws=ws, dA=db)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(torch_to_bits(da[:n]), torch_to_bits(db[:n]))
    assert gg.read_status(ws) == 0


# ------------------------------------------------------------------ activation and
# probability variants: QuickGeGLU, the weighted activation, the pre-FC1 multiply

@pytest.mark.parametrize("epi,act", [(1, "swiglu"), (3, "qgeglu")])
def test_gated_forward_variants(gg, epi, act):
    F, K = 320, 192
    rng = np.random.default_rng(91 + epi)
    E = len(COUNTS)
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 8
    X = normal_bf16(rng, (R_cap, K), 1.0)
    W1 = normal_bf16(rng, (E, 2 * F, K), 0.08)
    prob = rng.uniform(0.05, 1.0, R_cap).astype(np.float32)
    ws = gg.workspace(0, 1, E, "cuda")
    d_off = torch.from_numpy(off).cuda()
    d_prob = torch.from_numpy(prob).cuda()
    n = int(off[-1])
    h_ref = oracle.grouped_linear(oracle.bf16_bits_to_f64(X), W1, off)
    h_faith = oracle.round_to_bf16(h_ref)
    for weighted in (False, True):
        H1 = _nan_filled((R_cap, 2 * F))
        A = _nan_filled((R_cap, F))
        gg.grouped_fwd(bits_to_torch(X), bits_to_torch(W1), d_off, epi, ws=ws, C=A, H1_save=H1,
                       prob_of_row=d_prob if weighted else None)
        A2 = gg.glu(H1, d_off, E, epi, prob_of_row=d_prob if weighted else None,
                    A=_nan_filled((R_cap, F)))
        torch.cuda.synchronize()
        assert gg.read_status(ws) == 0
        p = prob.astype(np.float64)[:, None] if weighted else 1.0
        assert_parity(torch_to_f64(H1[:n]), h_ref[:n], "H1", faithful=h_faith[:n])
        ref = (p * oracle.glu(h_ref, act))[:n]
        assert_parity(torch_to_f64(A[:n]), ref, "A",
                      faithful=oracle.round_to_bf16(p * oracle.glu(h_faith, act))[:n])
        # fused epilogue and the standalone kernel round alike: bitwise equal
        np.testing.assert_array_equal(torch_to_bits(A[:n]), torch_to_bits(A2[:n]))
        assert np.all(torch_to_bits(A[n:]) == NAN_BF16)


@pytest.mark.parametrize("epi,act", [(2, "swiglu"), (4, "qgeglu")])
def test_gated_backward_variants(gg, epi, act):
    F, H = 320, 256
    rng = np.random.default_rng(97 + epi)
    E = len(COUNTS)
    off = _offsets(COUNTS)
    R_cap = int(off[-1]) + 16
    dY = normal_bf16(rng, (R_cap, H), 1.0)
    W2 = normal_bf16(rng, (E, H, F), 0.05)
    H1 = normal_bf16(rng, (R_cap, 2 * F), 1.5)
    prob = rng.uniform(0.05, 1.0, R_cap).astype(np.float32)
    ws = gg.workspace(0, 1, E, "cuda")
    nb, nbs = gg.rowdot_blocks(F), gg.rowdot_stride(F)
    rowdot = torch.full((R_cap, nbs), float("nan"), dtype=torch.float32, device="cuda")
    dH = _nan_filled((R_cap, 2 * F))
    gg.grouped_dgrad(bits_to_torch(dY), bits_to_torch(W2), torch.from_numpy(off).cuda(), epi,
                     H1=bits_to_torch(H1), prob_of_row=torch.from_numpy(prob).cuda(), ws=ws,
                     dA=dH, rowdot=rowdot)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    n = int(off[-1])
    acc = oracle.grouped_linear_t(oracle.bf16_bits_to_f64(dY), W2, off)
    h1 = oracle.bf16_bits_to_f64(H1)
    ref = oracle.glu_backward(prob.astype(np.float64)[:, None] * acc, h1, act)
    assert_parity(torch_to_f64(dH[:n]), ref[:n], "dH", faithful=oracle.round_to_bf16(ref[:n]))
    prod = acc * oracle.round_to_bf16(oracle.glu(h1, act))
    ref_rd = np.stack([prod[:, 128 * b:128 * (b + 1)].sum(axis=1) for b in range(nb)], axis=1)
    assert_parity(rowdot.cpu().numpy().astype(np.float64)[:n, :nb], ref_rd[:n], "rowdot")


def test_permute_rows_scaled_by_probability(gg):
    # the pre-FC1 multiply: dst[row] = bf16(prob * x) with the product in fp32,
    # bit-exact against the same fp32 product rounded on the host
    T, H, E, k, P = 300, 256, 8, 3, 16
    idx, prob = _permute_case(T, E, k, 33)
    rng = np.random.default_rng(5)
    x = normal_bf16(rng, (T, H), 1.0)
    p = gg.permute(bits_to_torch(x), torch.from_numpy(idx).cuda(), torch.from_numpy(prob).cuda(),
                   E, P)
    R_cap = p["Xp"].shape[0]
    dst = _nan_filled((R_cap, H))
    gg.permute_rows(bits_to_torch(x), p["row_of_slot"], p["slot_of_row"], p["offsets"], k, E, P,
                    R_cap, p["ws"], dst=dst, prob=torch.from_numpy(prob).cuda())
    torch.cuda.synchronize()
    assert gg.read_status(p["ws"]) == 0
    xv = oracle.bf16_bits_to_f64(x).astype(np.float32)
    ros = p["row_of_slot"].cpu().numpy().reshape(T, k)
    got = torch_to_f64(dst)
    for t in range(T):
        for j in range(k):
            want = oracle.round_to_bf16((np.float32(prob[t, j]) * xv[t]).astype(np.float64))
            np.testing.assert_array_equal(got[ros[t, j]], want)
    n = int(p["offsets"][-1].item())
    pad = p["slot_of_row"].cpu().numpy()[:n] < 0
    assert np.all(got[:n][pad] == 0)


@pytest.mark.parametrize("k", [3, 12])  # both register bounds of the kernel (8 and 32 slots)
def test_combine_dot_probability_gradient(gg, k):
    # dprob[t, j] = <dot_src[t], Yp[row(t, j)]>; the weighted sum itself is
    # bitwise the plain weighted combine
    T, H, R_cap = 300, 320, 4000
    rng = np.random.default_rng(43)
    rows = rng.permutation(R_cap)[:T * k].astype(np.int32)
    rows[[5, 77, 301]] = -1
    Yp = normal_bf16(rng, (R_cap, H), 1.0)
    xs = normal_bf16(rng, (T, H), 1.0)
    prob = rng.uniform(0, 1, (T, k)).astype(np.float32)
    ws = gg.workspace(T, k, 1, "cuda")
    d_rows = torch.from_numpy(rows).cuda()
    d_prob = torch.from_numpy(prob).cuda()
    out, dprob = gg.unpermute_combine(bits_to_torch(Yp), d_rows, d_prob, T, k, ws,
                                      dot_src=bits_to_torch(xs))
    out2 = gg.unpermute_combine(bits_to_torch(Yp), d_rows, d_prob, T, k, ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out2))
    y = oracle.bf16_bits_to_f64(Yp)
    ref = oracle.prob_grad(oracle.bf16_bits_to_f64(xs), y, rows, T, k)
    got = dprob.cpu().numpy().astype(np.float64)
    assert np.all(got.reshape(-1)[rows < 0] == 0)
    assert_parity(got, ref, "dprob (dot)")


@pytest.mark.parametrize("k", [8, 12])
@pytest.mark.parametrize("weighted", [False, True])
def test_combine_dot_with_separate_dot_rows(gg, k, weighted):
    # gg_unpermute_combine_dot: the sum runs over Sp while each pair's dot
    # takes its permuted row from a second tensor, dprob[t, j] =
    # <dot_src[t], D[row(t, j)]>; the sum is bitwise the plain combine of Sp
    T, H, R_cap = 300, 320, 4000
    rng = np.random.default_rng(47 + k)
    rows = rng.permutation(R_cap)[:T * k].astype(np.int32)
    rows[[5, 77, 301]] = -1
    Sp = normal_bf16(rng, (R_cap, H), 1.0)
    D = normal_bf16(rng, (R_cap, H), 1.0)
    xs = normal_bf16(rng, (T, H), 1.0)
    prob = rng.uniform(0, 1, (T, k)).astype(np.float32)
    ws = gg.workspace(T, k, 1, "cuda")
    d_rows = torch.from_numpy(rows).cuda()
    d_prob = torch.from_numpy(prob).cuda() if weighted else None
    out, dprob = gg.unpermute_combine_dot(bits_to_torch(Sp), d_rows, d_prob, T, k,
                                          bits_to_torch(xs), bits_to_torch(D), ws)
    out2 = gg.unpermute_combine(bits_to_torch(Sp), d_rows, d_prob, T, k, ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out2))
    ref = oracle.prob_grad(oracle.bf16_bits_to_f64(xs), oracle.bf16_bits_to_f64(D), rows, T, k)
    got = dprob.cpu().numpy().astype(np.float64)
    assert np.all(got.reshape(-1)[rows < 0] == 0)
    assert_parity(got, ref, "dprob (dot rows)")


@pytest.mark.parametrize("T,k,H", [(0, 4, 128), (7, 1, 64), (50, 32, 64), (129, 5, 576)])
def test_combine_dot_rows_edge_cases(gg, T, k, H):
    # an empty batch enqueues nothing; one slot; the 32-slot bound; a row of
    # 576 columns (the last pass leaves most lanes without a column group)
    R_cap = max(1, 3 * T * k)
    rng = np.random.default_rng(61 + T + k)
    rows = rng.permutation(R_cap)[:T * k].astype(np.int32)
    if T * k > 3:
        rows[1] = -1
    Sp = normal_bf16(rng, (R_cap, H), 1.0)
    D = normal_bf16(rng, (R_cap, H), 1.0)
    xs = normal_bf16(rng, (max(T, 1), H), 1.0)[:T]
    prob = rng.uniform(0, 1, (T, k)).astype(np.float32)
    ws = gg.workspace(max(T, 1), k, 1, "cuda")
    d_rows = torch.from_numpy(rows).cuda()
    d_prob = torch.from_numpy(prob).cuda()
    before = gg.launch_count()
    out, dprob = gg.unpermute_combine_dot(bits_to_torch(Sp), d_rows, d_prob, T, k,
                                          bits_to_torch(xs), bits_to_torch(D), ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    if T == 0:
        assert gg.launch_count() == before
        return
    out2 = gg.unpermute_combine(bits_to_torch(Sp), d_rows, d_prob, T, k, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out2))
    ref = oracle.prob_grad(oracle.bf16_bits_to_f64(xs), oracle.bf16_bits_to_f64(D), rows, T, k)
    got = dprob.cpu().numpy().astype(np.float64)
    assert np.all(got.reshape(-1)[rows < 0] == 0)
    assert_parity(got, ref, "dprob (dot rows, edge case)")
