"""Mimi RVQ dequantisation (pp_rvq_dequantize) against the oracle's, element by element
(GPU).  Codebooks are seeded N(0,1) fp32; codes are seeded uniform with closed-slot -1
rows and out-of-range codes mixed in."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

# Each output is a sum of <= 8 N(0,1) fp32 entries added in order in fp32, against the
# oracle's fp64 sum: the rounding error is below 8 * 2^-24 * sum|terms| < 1e-5.
TOL = 1e-5


def _codebooks(n_books, card, dim, seed):
    return synth.normal_f32(n_books * card * dim, seed, 31, 1.0).reshape(n_books, card, dim)


def _run(codes, stride, n_frames, cb, want_status=False):
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    n_books, card, dim = cb.shape
    dcodes = torch.from_numpy(np.ascontiguousarray(codes, np.int32)).cuda()
    dcb = torch.from_numpy(np.ascontiguousarray(cb)).cuda()
    out = torch.full((max(n_frames, 1), dim), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    pp.pp_rvq_dequantize(dcodes.data_ptr(), stride, n_frames, n_books, dcb.data_ptr(), card, dim,
                         out.data_ptr(), status.data_ptr() if want_status else None, stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()[:n_frames], int(status.item())


def _codes(n, n_books, card, seed):
    c = synth.uniform_i32(n * n_books, seed, 32, 0, card).reshape(n, n_books)
    return c


@pytest.mark.parametrize("dim", [4, 256, 512, 1028])
def test_rvq_matches_oracle(dim):
    n_books, card, n = 8, 2048, 37
    cb = _codebooks(n_books, card, dim, 5 + dim)
    codes = _codes(n, n_books, card, 7)
    codes[3, :] = -1                 # a closed slot
    codes[5, 2] = -1
    got, _ = _run(codes, n_books, n, cb)
    ref, bad = oracle.rvq_dequantize(codes, cb)
    assert bad == 0
    assert np.all(got[3] == 0)
    assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def test_rvq_reads_the_agent_rows_of_an_output_column():
    """codes = column + 1, stride 17: the agent rows 1..8 of a [B][17] tick column."""
    B, card, dim = 64, 2048, 512
    cb = _codebooks(8, card, dim, 9)
    col = synth.uniform_i32(B * 17, 11, 33, 0, card).reshape(B, 17)
    col[10, :] = -1                  # a closed slot's row of the column
    import torch
    import full_duplex_speech_lockstep_gb300 as pp
    dcol = torch.from_numpy(col).cuda()
    dcb = torch.from_numpy(cb).cuda()
    out = torch.empty((B, dim), dtype=torch.float32, device="cuda")
    pp.pp_rvq_dequantize(dcol.data_ptr() + 4, 17, B, 8, dcb.data_ptr(), card, dim, out.data_ptr(),
                         None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref, _ = oracle.rvq_dequantize(col[:, 1:9], cb)
    got = out.cpu().numpy()
    assert np.all(got[10] == 0)
    assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def test_rvq_out_of_range_codes_raise_index_status():
    cb = _codebooks(8, 64, 16, 13)
    codes = _codes(4, 8, 64, 15)
    got, st = _run(codes, 8, 4, cb, want_status=True)
    assert st == 0
    codes[2, 5] = 64
    got, st = _run(codes, 8, 4, cb, want_status=True)
    import full_duplex_speech_lockstep_gb300 as pp
    assert st & pp.PP_S_INDEX
    ref, bad = oracle.rvq_dequantize(codes, cb)
    assert bad == 1
    assert np.max(np.abs(got - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def test_rvq_large_batch_sampled():
    """65536 frames x 512 dims (a 5-minute-scale batch of 64 sessions); sampled frames."""
    n, card, dim = 65536, 2048, 512
    cb = _codebooks(8, card, dim, 17)
    codes = _codes(n, 8, card, 19)
    got, _ = _run(codes, 8, n, cb)
    rows = np.arange(0, n, 4093)
    ref, _ = oracle.rvq_dequantize(codes[rows], cb)
    assert np.max(np.abs(got[rows] - ref)) <= TOL * max(1.0, np.max(np.abs(ref)))


def test_rvq_rejects_bad_arguments():
    import full_duplex_speech_lockstep_gb300 as pp
    L = pp.lib()
    assert L.pp_rvq_dequantize(None, 8, 0, 8, None, 2048, 512, None, None, None) == pp.PP_OK
    assert L.pp_rvq_dequantize(None, 8, 1, 8, None, 2048, 512, None, None, None) == pp.PP_EINVAL
    assert L.pp_rvq_dequantize(None, 8, 1, 8, None, 2048, 510, None, None, None) == pp.PP_EINVAL
    assert L.pp_rvq_dequantize(None, 7, 1, 8, None, 2048, 512, None, None, None) == pp.PP_EINVAL
    assert L.pp_rvq_dequantize(None, 40, 1, 40, None, 2048, 512, None, None, None) == pp.PP_EINVAL
