"""The torch front end (bwd_gn3d_stats_gb300.nn): construction and argument checks (CPU)."""
import pytest
import torch

from bwd_gn3d_stats_gb300.nn import GroupNorm3d, group_norm_3d


def test_state_dict_matches_nn_groupnorm():
    ours, ref = GroupNorm3d(4, 16), torch.nn.GroupNorm(4, 16)
    assert list(ours.state_dict()) == list(ref.state_dict())
    ours.load_state_dict(ref.state_dict())  # a drop-in: the same keys and shapes
    none, ref_none = GroupNorm3d(4, 16, affine=False), torch.nn.GroupNorm(4, 16, affine=False)
    assert list(none.state_dict()) == list(ref_none.state_dict()) == []


def test_rejects_bad_configuration():
    with pytest.raises(ValueError):
        GroupNorm3d(3, 16)
    with pytest.raises(ValueError):
        GroupNorm3d(4, 16, activation="gelu")


def test_cpu_tensor_raises_no_cpu_path():
    x = torch.randn(1, 16, 2, 2, 2)
    with pytest.raises(RuntimeError, match="CUDA"):
        GroupNorm3d(4, 16)(x)
    with pytest.raises(RuntimeError, match="CUDA"):
        group_norm_3d(x, 4)
