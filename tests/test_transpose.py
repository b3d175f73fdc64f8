"""sgemm_transpose: out = in^T, bit for bit.

Host-side argument checks run without a GPU.  The GPU tests compare the
kernel's output with the oracle's transpose bit for bit (a transpose moves
values, so nothing is allowed to differ): ragged shapes over several CTA
blocks (128 rows x 32 columns each), the transpose page's 4096 x 4096 case,
padded and misaligned leading dimensions (the scalar path), special values,
untouched padding of the output, and the stream / launch-count contract.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp32_matrix_10_gb300 as sg

FAKE_IN, FAKE_OUT = 0x10000, 0x4000000


@pytest.fixture(scope="module")
def lib():
    from dense_fp32_matrix_10_gb300 import build
    l = ctypes.CDLL(build.build())
    l.sgemm_transpose.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    return l


# ------------------------------------------------------------------ host only
def test_bad_sizes_and_leading_dimensions(lib):
    t = lib.sgemm_transpose
    assert t(-1, 4, FAKE_IN, 4, FAKE_OUT, 4, None) == 1
    assert t(4, 5, FAKE_IN, 4, FAKE_OUT, 4, None) == 1        # ld_in < cols
    assert t(5, 4, FAKE_IN, 4, FAKE_OUT, 4, None) == 1        # ld_out < rows
    assert t(4, 4, 0, 4, FAKE_OUT, 4, None) == 1              # null input
    assert t(1 << 31, 4, FAKE_IN, 4, FAKE_OUT, 1 << 31, None) == 1


def test_overlap_and_in_place_are_aliasing(lib):
    t = lib.sgemm_transpose
    assert t(4, 4, FAKE_IN, 4, FAKE_IN, 4, None) == 2          # in place
    assert t(4, 4, FAKE_IN, 4, FAKE_IN + 60, 4, None) == 2      # last input element = first output
    assert t(4, 4, FAKE_IN, 4, FAKE_IN + 64, 4, None) in (0, 3)  # touching only


def test_empty_is_a_no_op(lib):
    assert lib.sgemm_transpose(0, 5, 0, 5, 0, 1, None) == 0
    assert lib.sgemm_transpose(5, 0, 0, 1, 0, 5, None) == 0
    assert lib.sgemm_last_launch_count() == 0


# ------------------------------------------------------------------ GPU
gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_10_gb300 import build
    build.build()
    torch.cuda.init()


def _bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def _input(rows, cols, seed, special=False):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(rows, cols, generator=g)
    if special:
        flat = X.view(-1)
        flat[::5] = -0.0
        flat[1::7] = float("inf")
        flat[2::11] = 1e-42
        flat.view(torch.int32)[3::13] = 0x7FC0ABCD     # NaN with a payload
    return X


def run_transpose(orc, rows, cols, seed=0, pad_in=0, pad_out=0, off_in=0, off_out=0, special=False):
    """GPU transpose of a rows x cols matrix stored with ld_in = cols + pad_in at
    element offset off_in (out likewise); checks bits against the oracle and
    that no element of the output buffer outside the result was written."""
    X = _input(rows, cols, seed, special)
    ld_in, ld_out = cols + pad_in, rows + pad_out
    hin = torch.full((off_in + rows * ld_in + 3,), float("nan"))
    hin[off_in: off_in + rows * ld_in].view(rows, ld_in)[:, :cols] = X
    din = hin.cuda()
    sentinel = 12345.0
    dout = torch.full((off_out + cols * ld_out + 3,), sentinel, device="cuda")
    sg.sgemm_transpose(rows, cols, din.data_ptr() + 4 * off_in, ld_in, dout.data_ptr() + 4 * off_out,
                       ld_out, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sg.sgemm_last_launch_count() == 1
    out = dout.cpu()
    res = out[off_out: off_out + cols * ld_out].view(cols, ld_out)[:, :rows].numpy()
    R = orc.transpose_f32(X.numpy())
    assert np.array_equal(_bits(res), _bits(R)), f"{rows}x{cols}"
    mask = torch.ones_like(out, dtype=torch.bool)
    mask[off_out: off_out + cols * ld_out].view(cols, ld_out)[:, :rows] = False
    assert bool(torch.all(out[mask] == sentinel)), "written outside the result"


SHAPES = [(1, 1), (1, 7), (7, 1), (5, 3), (33, 17), (127, 129), (128, 32), (129, 33), (300, 260),
          (1000, 1013), (8192, 64), (64, 8192), (4096, 4096)]


@gpu
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{r}x{c}" for r, c in SHAPES])
def test_shapes_bit_exact(_cuda, orc, shape):
    run_transpose(orc, *shape, seed=sum(shape))


@gpu
def test_special_values_bit_exact(_cuda, orc):
    run_transpose(orc, 260, 300, seed=1, special=True)      # vector path
    run_transpose(orc, 61, 37, seed=2, special=True)        # scalar edges


@gpu
@pytest.mark.parametrize("pads", [(4, 4, 0, 0), (3, 5, 0, 0), (0, 0, 1, 3), (8, 0, 2, 0)],
                         ids=["padded_aligned", "padded_odd", "offset", "mixed"])
def test_leading_dimensions_and_offsets(_cuda, orc, pads):
    pi, po, oi, oo = pads
    run_transpose(orc, 200, 136, seed=3, pad_in=pi, pad_out=po, off_in=oi, off_out=oo)


@gpu
@pytest.mark.parametrize("rows", [201, 202, 203])
def test_ragged_output_rows_keep_padding(_cuda, orc, rows):
    """Aligned buffers whose output rows (`rows` floats) do not end on a
    16-byte boundary: the padding after each output row stays untouched (a
    TMA store would write the rest of the row's last 16-byte granule)."""
    run_transpose(orc, rows, 136, seed=rows, pad_out=(-rows) % 4 + 4)


@gpu
def test_torch_wrapper_and_stream(_cuda, orc):
    s = torch.cuda.Stream()
    X = torch.randn(513, 257, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        Y = sg.transpose(X, stream=s)
    s.synchronize()
    assert np.array_equal(_bits(Y.cpu().numpy()), _bits(orc.transpose_f32(X.cpu().numpy())))
    # a view with a longer row as the output
    big = torch.zeros(257, 600, device="cuda")
    sg.transpose(X, out=big[:, :513])
    torch.cuda.synchronize()
    assert np.array_equal(_bits(big[:, :513].cpu().numpy()), _bits(orc.transpose_f32(X.cpu().numpy())))
    assert torch.all(big[:, 513:] == 0)


@gpu
def test_large_by_structure(_cuda):
    """16384 x 8192 (512 MiB each way), every output checked on the GPU by a
    property: input element (r, c) holds the exact key (r mod 4096) * 4096 +
    (c mod 4096) (below 2^24, so exact in FP32), and output element (c, r) must
    hold that key, built independently from the output's own indices."""
    rows, cols = 16384, 8192
    r = torch.arange(rows, device="cuda").view(-1, 1)
    c = torch.arange(cols, device="cuda").view(1, -1)
    X = ((r % 4096) * 4096 + (c % 4096)).to(torch.float32)
    Y = sg.transpose(X)
    torch.cuda.synchronize()
    del X
    oc = torch.arange(cols, device="cuda").view(-1, 1)     # output row = input column
    orr = torch.arange(rows, device="cuda").view(1, -1)    # output column = input row
    expect = ((orr % 4096) * 4096 + (oc % 4096)).to(torch.float32)
    assert torch.equal(Y, expect)
