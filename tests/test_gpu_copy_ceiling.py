"""softmax_rows_copy_ceiling, the bench's copy ceiling: it copies exactly the
valid bytes of every row, at any pitches, aligned or not, and leaves the pad
bytes of the output rows alone."""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("M,row_bytes,ld_in,ld_out,off_in,off_out", [
    (1, 16, 16, 16, 0, 0),
    (16384, 2000, 2048, 2000, 0, 0),      # the padded bf16 workload's rows
    (1024, 1024, 1024, 1024, 0, 0),
    (3, 262144, 262144, 262160, 0, 16),
    (37, 4097 * 2, 4097 * 2, 4100 * 2, 2, 6),  # unaligned: the byte path
    (5, 1, 3, 7, 1, 5),
    # Co-aligned (equal base offsets and pitches modulo 16): head, vectors, tail.
    (128, 32769 * 2, 32769 * 2, 32769 * 2, 0, 0),  # the f16 128 x 32769 rows
    (7, 100, 130, 146, 3, 3),
    (4, 10, 18, 34, 5, 5),                          # rows shorter than their head
    (3, 40, 40, 56, 9, 9),
    (9, 333, 338, 354, 14, 14),
])
def test_copies_rows_exactly(M, row_bytes, ld_in, ld_out, off_in, off_out):
    g = torch.Generator().manual_seed(M * 7 + row_bytes)
    src = torch.randint(0, 256, (off_in + M * ld_in,), dtype=torch.uint8, generator=g).cuda()
    dst = torch.full((off_out + M * ld_out + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_copy_ceiling(src.data_ptr() + off_in, dst.data_ptr() + off_out, M, row_bytes,
                                 ld_in, ld_out)
    torch.cuda.synchronize()
    s = src.cpu().numpy()[off_in:].reshape(M, ld_in)
    d = dst.cpu().numpy()
    body = d[off_out:off_out + M * ld_out].reshape(M, ld_out)
    assert np.array_equal(body[:, :row_bytes], s[:, :row_bytes])
    assert (body[:, row_bytes:] == 0xA5).all()
    assert (d[:off_out] == 0xA5).all() and (d[off_out + M * ld_out:] == 0xA5).all()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


@pytest.mark.parametrize("M,row_bytes,ld_a,ld_b,ld_out,off", [
    (64, 262144, 262144, 262144, 262144, 0),    # the backward's few wide rows, f16
    (100, 8192, 8208, 8192, 8224, 0),
    (9, 333, 340, 350, 360, 3),                 # unaligned: the byte path
])
def test_pair_ceiling_xors_rows_exactly(M, row_bytes, ld_a, ld_b, ld_out, off):
    g = torch.Generator().manual_seed(M + row_bytes)
    a = torch.randint(0, 256, (off + M * ld_a,), dtype=torch.uint8, generator=g).cuda()
    b = torch.randint(0, 256, (off + M * ld_b,), dtype=torch.uint8, generator=g).cuda()
    o = torch.full((off + M * ld_out + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_copy_ceiling2(a.data_ptr() + off, b.data_ptr() + off, o.data_ptr() + off, M,
                                  row_bytes, ld_a, ld_b, ld_out)
    torch.cuda.synchronize()
    ah = a.cpu().numpy()[off:].reshape(M, ld_a)[:, :row_bytes]
    bh = b.cpu().numpy()[off:].reshape(M, ld_b)[:, :row_bytes]
    oh = o.cpu().numpy()
    body = oh[off:off + M * ld_out].reshape(M, ld_out)
    assert np.array_equal(body[:, :row_bytes], ah ^ bh)
    assert (body[:, row_bytes:] == 0xA5).all() and (oh[off + M * ld_out:] == 0xA5).all()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
