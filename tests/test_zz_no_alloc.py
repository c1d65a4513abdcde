"""pp_ring_attention_noalloc: the ring attention for callers that cannot allocate device
memory (a host whose memory belongs to a pooling allocator, a real-time frame loop that
must not allocate).  Through the C ABI it must give the same output as
pp_ring_attention with caller scratch, within the attention tests' tolerance, on two
calls in a row (the built-in scratch keeps the previous call's contents).  This file is
collected last so that a failure here stops a run only after every other test ran."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

TOL = 1e-4   # the tolerance of the ring-attention tests


def _inputs(B, H, D, W, seed):
    import torch
    k = synth.normal_bf16(B * H * W * D, seed, 1, 1.0)
    v = synth.normal_bf16(B * H * W * D, seed, 2, 1.0)
    q = synth.normal_f32(B * H * D, seed, 3, 1.0)
    n = np.array([W, 0, 1, W // 3 + 5, W - 1, 17][:B] + [W] * max(0, B - 6), np.int32)
    return (torch.from_numpy(q).cuda(), torch.from_numpy(k.view(np.int16)).cuda(),
            torch.from_numpy(v.view(np.int16)).cuda(), torch.from_numpy(n).cuda())


@pytest.mark.parametrize("B,H,D,W", [(6, 3, 64, 700), (64, 32, 128, 3000)])
def test_noalloc_matches_scratch_entry_point(B, H, D, W):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    q, k, v, n = _inputs(B, H, D, W, 31 + D)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((B, H * D), dtype=torch.float32, device="cuda")
    nbytes = pp.pp_ring_attention_scratch_bytes(B, H, D, W)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    pp.pp_ring_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), H * W * D, n.data_ptr(),
                         B, H, D, W, ref.data_ptr(), scratch.data_ptr(), nbytes, stream)
    for call in range(2):
        out = torch.full((B, H * D), float("nan"), dtype=torch.float32, device="cuda")
        pp.pp_ring_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), H * W * D,
                                     n.data_ptr(), B, H, D, W, out.data_ptr(), stream)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy(), ref.cpu().numpy()
        assert np.all(np.isfinite(a)), call
        assert np.max(np.abs(a - b)) <= TOL * max(1.0, float(np.max(np.abs(b)))), call


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import full_duplex_speech_lockstep_gb300 as pp
    for B, H, D, W in [(65, 32, 128, 100), (1, 1, 64, 3073)]:
        with pytest.raises(pp.PPError) as e:
            pp.pp_ring_attention_noalloc(0, 0, 0, 0, 0, B, H, D, W, 0, None)
        assert e.value.code == pp.PP_E_RANGE
