"""The tick's split-K ring attention as a standalone call (pp_ring_attention) against the
CPU oracle's attention, per slot and head (GPU)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

# fp32 scores and accumulation over at most a few thousand bf16 keys against the fp64
# oracle: |error| stays far below 1e-4 of the largest |V| entry.
TOL = 1e-4


def _run(B, H, D, W, n_valid, seed):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    k = synth.normal_bf16(B * H * W * D, seed, 1, 1.0).reshape(B, H, W, D)
    v = synth.normal_bf16(B * H * W * D, seed, 2, 1.0).reshape(B, H, W, D)
    q = synth.normal_f32(B * H * D, seed, 3, 1.0).reshape(B, H, D)
    dk = torch.from_numpy(k.view(np.int16)).cuda()
    dv = torch.from_numpy(v.view(np.int16)).cuda()
    dq = torch.from_numpy(q).cuda()
    dn = torch.from_numpy(np.asarray(n_valid, np.int32)).cuda()
    out = torch.full((B, H * D), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = pp.pp_ring_attention_scratch_bytes(B, H, D, W)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):   # the second call must find its scratch reusable as left
        pp.pp_ring_attention(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), H * W * D,
                             dn.data_ptr(), B, H, D, W, out.data_ptr(), status.data_ptr(),
                             scratch.data_ptr(), nbytes, stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0   # no bounded wait gave up
    return q, k, v, out.cpu().numpy().reshape(B, H, D)


@pytest.mark.parametrize("D,W", [(32, 40), (64, 600), (128, 777)])
def test_ring_attention_matches_oracle(D, W):
    B, H = 5, 3
    n_valid = [W, 0, 1, W // 2 + 3, min(256, W - 1)]
    q, k, v, got = _run(B, H, D, W, n_valid, 7 + D)
    for s in range(B):
        for h in range(H):
            if n_valid[s] == 0:
                assert np.all(got[s, h] == 0)
                continue
            ref = oracle.attend(q[s, h], k[s, h], v[s, h], min(n_valid[s], W))
            assert np.max(np.abs(got[s, h] - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def _check_all(q, k, v, got, n_valid, W):
    for s in range(got.shape[0]):
        n = min(n_valid[s], W)
        for h in range(got.shape[1]):
            if n <= 0:
                assert np.all(got[s, h] == 0), (s, h)
                continue
            ref = oracle.attend(q[s, h], k[s, h], v[s, h], n)
            err = np.max(np.abs(got[s, h] - ref))
            assert err <= TOL * max(1.0, np.max(np.abs(ref))), (s, h, n, err)


def test_ring_attention_full_size():
    """B=64 slots x 32 heads x 128 over full 3000-position rings (the bench workload's
    attention): every (slot, head) against the oracle."""
    B, H, D, W = 64, 32, 128, 3000
    n_valid = [W] * B
    q, k, v, got = _run(B, H, D, W, n_valid, 11)
    _check_all(q, k, v, got, n_valid, W)


def test_ring_attention_full_size_ragged():
    """B=64 at W=3000 with a seeded mix of valid lengths: ragged last chunks, one-key
    and closed slots, lengths on and next to chunk edges, and lengths above W."""
    B, H, D, W = 64, 32, 128, 3000
    edges = [0, 1, 2, 127, 128, 129, 255, 256, 2943, 2944, 2945, 2999, 3000, 3001, 9000]
    rnd = synth.uniform_i32(B - len(edges), 19, 1, 1, W + 1).tolist()
    n_valid = edges + rnd
    q, k, v, got = _run(B, H, D, W, n_valid, 23)
    _check_all(q, k, v, got, n_valid, W)


def test_ring_attention_clamps_valid_lengths():
    """n_valid above the window counts as the window; negative counts as closed."""
    B, H, D, W = 3, 2, 64, 300
    q, k, v, got = _run(B, H, D, W, [W + 500, -4, W], 21)
    assert np.all(got[1] == 0)
    for h in range(H):
        assert np.array_equal(got[0, h], got[0, h])
        ref = oracle.attend(q[0, h], k[0, h], v[0, h], W)
        assert np.max(np.abs(got[0, h] - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def test_ring_attention_rejects_bad_arguments():
    import full_duplex_speech_lockstep_gb300 as pp
    with pytest.raises(pp.PPError):
        pp.pp_ring_attention_scratch_bytes(4, 2, 48, 100)
    with pytest.raises(pp.PPError):
        pp.pp_ring_attention(0, 0, 0, 0, 0, 1, 1, 64, 10, 0, 0, 0, 0, None)
