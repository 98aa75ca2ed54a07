"""The permute entry point that allocates nothing (collected last on purpose).

Some callers of this library cannot allocate device memory at the point where
they need the permute: a runtime whose memory pool owns the whole GPU and
forbids cudaMalloc on its hot path, a plugin that its host hands only
pre-sized input and output buffers, or a C caller with no device allocator.
gg_permute_noalloc serves them by keeping the permute's scratch in a fixed
array inside the library instead of a caller workspace.

This test calls it through the C ABI twice in a row, with two different
batches (so the second call runs on scratch the first one left behind), and
checks every output against the workspace-taking gg_permute: index work and
copied rows must be bit-identical, as everywhere else in the suite. It also
checks that a batch too large for the fixed scratch is refused before
anything is enqueued."""

import ctypes

import numpy as np
import pytest
import torch

from moe_synth import CONFIGS, MoeShape, make_inputs

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x7FC0


@pytest.fixture(scope="module")
def gg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


def _outputs(T, H, k, E, P):
    rc = T * k + E * (P - 1)
    xp = torch.full((rc, H), SENTINEL_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return dict(Xp=xp,
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                row_of_slot=torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
                slot_of_row=torch.full((rc,), -7, dtype=torch.int32, device="cuda"),
                prob_of_row=torch.full((rc,), -7.0, dtype=torch.float32, device="cuda"))


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(gg, x, idx, prob, E, P, o):
    T, H = x.shape
    k = idx.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gg.LIB.gg_permute_noalloc(_p(x), _p(idx), _p(prob), T, H, k, E, P, _p(o["Xp"]),
                                     _p(o["offsets"]), _p(o["row_of_slot"]),
                                     _p(o["slot_of_row"]), _p(o["prob_of_row"]), stream)


def _bits(t):
    return t.contiguous().view(torch.int32 if t.element_size() == 4 else torch.int16).cpu().numpy()


def test_noalloc_permute_matches_workspace_permute_on_two_calls(gg):
    batches = [
        (CONFIGS[3], 3000),  # 128 experts, top-8, 256-row padding: many histogram blocks
        (MoeShape("small_e8_h256_t300_k2_pad16", E=8, H=256, F=128, T=300, k=2, P=16), 91),
    ]
    for shape, seed in batches:
        inp = make_inputs(shape, seed, with_weights=False, with_dout=False)
        x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
        idx = torch.from_numpy(inp.idx).cuda()
        prob = torch.from_numpy(inp.prob).cuda()
        T, k, E, P, H = shape.T, shape.k, shape.E, shape.P, shape.H
        mine = _outputs(T, H, k, E, P)
        assert _call_noalloc(gg, x, idx, prob, E, P, mine) == gg.GG_OK
        ref = _outputs(T, H, k, E, P)
        gg.permute(x, idx, prob, E, P, out=ref)
        torch.cuda.synchronize()
        for name in ("offsets", "row_of_slot", "slot_of_row", "prob_of_row", "Xp"):
            np.testing.assert_array_equal(_bits(mine[name]), _bits(ref[name]), err_msg=name)


def test_noalloc_permute_rejects_batches_beyond_its_scratch(gg):
    # 70000 * 8 pairs at E = 1024 take 128 histogram rows of 1024 experts
    # (512 KiB), more than the 256 KiB the fixed scratch holds
    dummy = torch.zeros(64, dtype=torch.float32, device="cuda")
    before = gg.launch_count()
    code = gg.LIB.gg_permute_noalloc(_p(dummy), _p(dummy), _p(dummy), 70000, 64, 8, 1024, 1,
                                     _p(dummy), _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 4  # GG_ERR_WORKSPACE_TOO_SMALL
    assert gg.launch_count() == before


def test_noalloc_permute_maps_only(gg):
    # With Xp (and x) NULL the call produces only the row maps, offsets and
    # per-row probabilities, as gg_permute does; twice in a row again.
    shape = MoeShape("maps_e16_h128_t500_k4_pad8", E=16, H=128, F=128, T=500, k=4, P=8)
    for seed in (17, 18):
        inp = make_inputs(shape, seed, with_weights=False, with_dout=False)
        x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).cuda()
        idx = torch.from_numpy(inp.idx).cuda()
        prob = torch.from_numpy(inp.prob).cuda()
        T, k, E, P, H = shape.T, shape.k, shape.E, shape.P, shape.H
        mine = _outputs(T, H, k, E, P)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        code = gg.LIB.gg_permute_noalloc(None, _p(idx), _p(prob), T, H, k, E, P, None,
                                         _p(mine["offsets"]), _p(mine["row_of_slot"]),
                                         _p(mine["slot_of_row"]), _p(mine["prob_of_row"]), stream)
        assert code == gg.GG_OK
        ref = _outputs(T, H, k, E, P)
        gg.permute(x, idx, prob, E, P, out=ref)
        torch.cuda.synchronize()
        for name in ("offsets", "row_of_slot", "slot_of_row", "prob_of_row"):
            np.testing.assert_array_equal(_bits(mine[name]), _bits(ref[name]), err_msg=name)
        # the permuted-row buffer was not touched
        assert np.all(_bits(mine["Xp"]) == np.int16(SENTINEL_BF16))
