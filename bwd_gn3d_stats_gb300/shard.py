"""GroupNorm of a volume split into shards (spatial sharding, one D-slab per
rank): the whole volume's statistics from one exchange per direction.

Each rank holds its slab as a contiguous [N, C, D_k, H, W] tensor.  The forward
exchanges every rank's per-group moments (count, mean, M2) and combines them in
rank order; the backward exchanges the per-row sums (sum dy, sum dy*(x - mean))
and adds them in rank order.  Every arithmetic step runs in libgn3d's kernels
(gn3d_forward_moments, gn3d_moments_combine, gn3d_forward_apply,
gn3d_backward_sums, gn3d_sums_combine, gn3d_backward_dx_from_sums); this module
marshals arguments and gathers the partial results over a torch.distributed
process group in rank order.  Without an initialized process group (or with one
rank) the exchange is the identity and the results equal gn3d_forward /
gn3d_backward on the tensor bit for bit.
"""
from __future__ import annotations

from . import BF16, F32, _dtype_code, _ptr, _shape5, gn3d_backward_dx_from_sums, gn3d_backward_sums, \
    gn3d_forward_apply, gn3d_forward_moments, gn3d_moments_combine, gn3d_sums_combine

MOMENT_BYTES = 24  # gn3d_moments: int64 count, then mean_hi, mean_lo, m2, reserved (fp32)


def all_gather_rank_order(t, group=None):
    """[world, *t.shape]: every rank's tensor, stacked in rank order (the
    tensor itself, unsqueezed, without a process group or with one rank)."""
    import torch

    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return t.unsqueeze(0)
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def _stream(t):
    import torch

    return torch.cuda.current_stream(t.device).cuda_stream


def moments(x, G: int):
    """Per group moments of x (a shard), as raw gn3d_moments records: uint8 [N*G*24]."""
    import torch

    N, C, D, H, W = _shape5(x)
    m = torch.empty(N * G * MOMENT_BYTES, dtype=torch.uint8, device=x.device)
    gn3d_forward_moments(x.data_ptr(), N, C, D, H, W, G, _dtype_code(x.dtype), m.data_ptr(), _stream(x))
    return m


def combine_moments(stacked):
    """[K, N*G*24] moments of K shards (rank order) -> the combined [N*G*24]."""
    import torch

    K = stacked.shape[0]
    ng = stacked.shape[1] // MOMENT_BYTES
    out = torch.empty(ng * MOMENT_BYTES, dtype=torch.uint8, device=stacked.device)
    gn3d_moments_combine(stacked.contiguous().data_ptr(), K, ng, out.data_ptr(), _stream(stacked))
    return out


def moment_counts(m):
    """The count field of each record (int64 [N*G])."""
    return m.view(-1, MOMENT_BYTES)[:, :8].contiguous().view(-1).view(__import__("torch").int64)


def forward_apply(x, gamma, beta, G: int, m, eps: float = 1e-5, out_dtype=None):
    """y, mean, rstd of a shard normalized with the whole volume's moments m."""
    import torch

    N, C, D, H, W = _shape5(x)
    out_dtype = x.dtype if out_dtype is None else out_dtype
    y = torch.empty((N, C, D, H, W), dtype=out_dtype, device=x.device)
    mean = torch.empty((N, G), dtype=torch.float32, device=x.device)
    rstd = torch.empty((N, G), dtype=torch.float32, device=x.device)
    gn3d_forward_apply(x.data_ptr(), _ptr(gamma), _ptr(beta), N, C, D, H, W, G, float(eps), _dtype_code(x.dtype),
                       _dtype_code(out_dtype), m.data_ptr(), y.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                       _stream(x))
    return y, mean, rstd


def backward_sums(dy, x, mean, rstd, G: int):
    """Per row (n, c) of a shard: (sum dy, sum dy*(x - mean)) as float32 [N*C*2]."""
    import torch

    N, C, D, H, W = _shape5(x)
    s = torch.empty(N * C * 2, dtype=torch.float32, device=x.device)
    gn3d_backward_sums(dy.contiguous().data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), N, C, D, H, W, G,
                       _dtype_code(x.dtype), s.data_ptr(), _stream(x))
    return s


def combine_sums(stacked):
    """[K, N*C*2] row sums of K shards (rank order) -> their totals [N*C*2]."""
    import torch

    K = stacked.shape[0]
    nc = stacked.shape[1] // 2
    out = torch.empty(nc * 2, dtype=torch.float32, device=stacked.device)
    gn3d_sums_combine(stacked.contiguous().data_ptr(), K, nc, out.data_ptr(), _stream(stacked))
    return out


def backward_dx_from_sums(dy, x, mean, rstd, gamma, G: int, sums, group_count: int):
    """dx, dgamma, dbeta of a shard from the whole volume's row sums (groups of
    group_count elements)."""
    import torch

    N, C, D, H, W = _shape5(x)
    dx = torch.empty_like(x)
    dgamma = torch.empty((C,), dtype=torch.float32, device=x.device)
    dbeta = torch.empty((C,), dtype=torch.float32, device=x.device)
    gn3d_backward_dx_from_sums(dy.contiguous().data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                               _ptr(gamma), sums.data_ptr(), int(group_count), N, C, D, H, W, G,
                               _dtype_code(x.dtype), dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), _stream(x))
    return dx, dgamma, dbeta


def forward_sharded(x, gamma, beta, G: int, eps: float = 1e-5, out_dtype=None, group=None):
    """The forward of this rank's shard with the whole volume's statistics:
    (y, mean, rstd, group_count)."""
    m = combine_moments(all_gather_rank_order(moments(x, G), group))
    y, mean, rstd = forward_apply(x, gamma, beta, G, m, eps, out_dtype)
    return y, mean, rstd, int(moment_counts(m)[0].item()) if m.numel() else 0


def backward_sharded(dy, x, mean, rstd, gamma, G: int, group_count: int, group=None):
    """The backward of this rank's shard at the whole volume's statistics."""
    total = combine_sums(all_gather_rank_order(backward_sums(dy, x, mean, rstd, G), group))
    return backward_dx_from_sums(dy, x, mean, rstd, gamma, G, total, group_count)


__all__ = ["MOMENT_BYTES", "all_gather_rank_order", "moments", "combine_moments", "moment_counts",
           "forward_apply", "backward_sums", "combine_sums", "backward_dx_from_sums", "forward_sharded",
           "backward_sharded", "BF16", "F32"]
