"""The guard-band helper the GPU tests wrap their outputs in catches a write
just outside the tensor on either side, and leaves the tensor itself usable."""
import torch

from helpers import GUARD_BYTES, Guarded, guarded_like


def test_untouched_guards_pass():
    g = Guarded((7, 9), torch.bfloat16, device="cpu")
    assert torch.isnan(g.t.float()).all()  # unwritten elements show up as NaN
    g.t.fill_(2.0)
    g.check("filled")


def test_write_past_the_end_is_caught():
    g = Guarded((5, 3), torch.float32, device="cpu")
    g.buf[GUARD_BYTES + g.nbytes] = 0  # the first byte after the tensor
    try:
        g.check("past end")
    except AssertionError as e:
        assert "after: False" in str(e)
    else:
        raise AssertionError("an overrun past the end went unnoticed")


def test_write_before_the_start_is_caught():
    g = guarded_like(torch.zeros(4, 4))
    g.buf[GUARD_BYTES - 1] ^= 0xFF  # the last byte before the tensor
    try:
        g.check("before start")
    except AssertionError as e:
        assert "before intact: False" in str(e)
    else:
        raise AssertionError("an underrun before the start went unnoticed")


def test_tensor_view_is_aligned_and_sized():
    g = Guarded((3, 256), torch.bfloat16, device="cpu", fill=None)
    assert g.t.data_ptr() % 16 == 0
    assert g.nbytes == 3 * 256 * 2
    assert g.t.shape == (3, 256)
