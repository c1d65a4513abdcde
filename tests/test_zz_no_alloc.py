"""pp_ring_attention_noalloc: the ring attention for callers that cannot allocate device
memory (a host whose memory belongs to a pooling allocator, a real-time frame loop that
must not allocate).  Through the C ABI it must give the same output as
pp_ring_attention with caller scratch: both launch the same kernels with the same
reduction order, so the outputs are compared bit for bit (which is within the ring
attention tests' 1e-4 tolerance).  The built-in scratch keeps the previous call's
contents, so calls follow each other in a row and at changing sizes: a smaller call
after a larger one must not be disturbed by the larger call's leftovers.  This file is
collected last so that a failure here stops a run only after every other test ran."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _inputs(B, H, D, W, seed, n_valid=None):
    """Ring K/V (bf16 N(0,1), generated on the device), queries and valid lengths."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    lib = synth._dev_lib()
    kv = []
    for sid in (1, 2):
        t = torch.empty(B * H * W * D, dtype=torch.int16, device="cuda")
        assert lib.ppsyn_normal_bf16_dev(t.data_ptr(), t.numel(), 0, seed, sid,
                                         synth.normal_scale(1.0), stream) == 0
        kv.append(t)
    q = synth.normal_f32(B * H * D, seed, 3, 1.0)
    if n_valid is None:
        n_valid = [W, 0, 1, W // 3 + 5, W - 1, 17][:B] + [W] * max(0, B - 6)
    n = np.asarray(n_valid, np.int32)
    return torch.from_numpy(q).cuda(), kv[0], kv[1], torch.from_numpy(n).cuda()


def _status():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _with_scratch(q, k, v, n, B, H, D, W):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.full((B, H * D), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    nbytes = pp.pp_ring_attention_scratch_bytes(B, H, D, W)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    pp.pp_ring_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), H * W * D, n.data_ptr(),
                         B, H, D, W, out.data_ptr(), st.data_ptr(), scratch.data_ptr(), nbytes,
                         stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.cpu().numpy()


def _without_scratch(q, k, v, n, B, H, D, W):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.full((B, H * D), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    pp.pp_ring_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), H * W * D,
                                 n.data_ptr(), B, H, D, W, out.data_ptr(), st.data_ptr(),
                                 stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("B,H,D,W", [(6, 3, 64, 700), (64, 32, 128, 3000)])
def test_noalloc_matches_scratch_entry_point(B, H, D, W):
    args = _inputs(B, H, D, W, 31 + D) + (B, H, D, W)
    ref = _with_scratch(*args)
    for call in range(2):
        got = _without_scratch(*args)
        assert np.all(np.isfinite(got)), call
        assert np.array_equal(got, ref), call


@pytest.mark.parametrize("D", [64, 128])
def test_noalloc_after_a_larger_call(D):
    """A large call fills most of the built-in scratch (partials and tickets); a smaller
    call with another slot count, window and valid lengths follows, then the large one
    again: each equals the caller-scratch entry point on the same inputs."""
    big = (32, 64, D, 3000) if D == 128 else (48, 40, D, 3000)
    small = (5, 7, D, 333)
    a_big = _inputs(*big, seed=41 + D, n_valid=[3000 - 7 * i for i in range(big[0])])
    a_small = _inputs(*small, seed=43 + D, n_valid=[333, 129, 128, 1, 0])
    ref_big = _with_scratch(*a_big, *big)
    ref_small = _with_scratch(*a_small, *small)
    assert np.array_equal(_without_scratch(*a_big, *big), ref_big)
    assert np.array_equal(_without_scratch(*a_small, *small), ref_small)
    assert np.array_equal(_without_scratch(*a_big, *big), ref_big)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import full_duplex_speech_lockstep_gb300 as pp
    for B, H, D, W in [(65, 32, 128, 100), (1, 1, 64, 3073)]:
        with pytest.raises(pp.PPError) as e:
            pp.pp_ring_attention_noalloc(0, 0, 0, 0, 0, B, H, D, W, 0, 0, None)
        assert e.value.code == pp.PP_E_RANGE
