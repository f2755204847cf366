"""Host-side checks of the layer object that need no GPU: the token tensors it hands to the library
as bare pointers are checked for shape, dtype and layout before any launch."""
import pytest
import torch

from sparse_moe_fine_gb300.layer import MoELayer


def _bare_layer(T=8, H=16, dtype=torch.bfloat16):
    L = MoELayer.__new__(MoELayer)  # only the fields the check reads
    L.T, L.H, L.dtype = T, H, dtype
    return L


def test_token_check_rejects_wrong_shape_and_dtype():
    L = _bare_layer()
    with pytest.raises(ValueError, match="x: expected a \\[8, 16\\]"):
        L._check_tokens(x=torch.zeros(8, 17, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="dy: expected"):
        L._check_tokens(x=None, dy=torch.zeros(16, 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="y: expected"):
        L._check_tokens(y=torch.zeros(8, 16, dtype=torch.float32))


def test_token_check_rejects_host_and_strided_tensors():
    L = _bare_layer()
    # right shape and dtype, but host memory: the library would read it as a device address
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        L._check_tokens(x=torch.zeros(8, 16, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="contiguous CUDA tensor"):
        L._check_tokens(dx=torch.zeros(16, 8, dtype=torch.bfloat16).t())


def test_token_check_skips_absent_outputs():
    _bare_layer()._check_tokens(x=None, y=None, dx=None)
