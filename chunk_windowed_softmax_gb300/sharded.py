"""Head-sharded (Ulysses-style) use of the library across the ranks of a ``torch.distributed`` group.

The MiniMax-H3 Ulysses pull request (sglang #43164, Motivation and Modifications item 4: 56 heads split over the
ranks) runs attention on several GPUs by exchanging q, k and v so that each rank holds the whole sequence for a
subset of the heads, and by exchanging the output back; the VDN-Minimax-H3 window-attention article (section 四)
deploys the decomposed path that way on 8 GPUs. Every (b, h) slice of the window attention is independent of the
others, so a rank computes its heads with an ordinary plan on its own GPU (the library's kernels) and the only
cross-rank steps are the two all-to-all exchanges below; there is no halo and no cross-rank softmax merge.

Layouts (B, H, D and the packed sequence of L = T*S + G rows as everywhere in the library):
  * sequence shard: rank p holds the rows [off_p, off_p + n_p) of every head as a [B, n_p, H, D] tensor, where
    ``seq_sizes`` = [n_0, ..., n_{N-1}] sums to L (``even_seq_sizes`` splits L as evenly as possible);
  * head shard: rank p holds the heads [p H/N, (p + 1) H/N) of every row as a [B, L, H/N, D] tensor (H must be a
    multiple of N).
The exchanges are ``torch.distributed.all_to_all_single`` calls (NCCL between GPUs, gloo on the CPU); this module
only arranges the blocks around them. A head range of tensors that hold every head needs no exchange at all:
``forward_heads`` runs a plan whose layout has H = nh and the full tensors' strides on pointers advanced by
h0 * stride_h (the layout rule of ``include/wa.h``).
"""
import torch
import torch.distributed as dist


def even_seq_sizes(L, world):
    """Split L rows into `world` consecutive shards whose sizes differ by at most one (the first ones larger)."""
    base, extra = divmod(L, world)
    return [base + (1 if p < extra else 0) for p in range(world)]


def _world(group):
    return dist.get_world_size(group) if dist.is_initialized() else 1


def _rank(group):
    return dist.get_rank(group) if dist.is_initialized() else 0


def seq_to_heads(x, seq_sizes, group=None):
    """This rank's sequence shard [B, n_rank, H, D] -> its head shard [B, L, H/N, D] (one all-to-all)."""
    world, rank = _world(group), _rank(group)
    B, n, H, D = x.shape
    if world == 1:
        return x.contiguous()
    if H % world:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    if n != seq_sizes[rank] or len(seq_sizes) != world:
        raise ValueError("the shard does not match seq_sizes")
    hn = H // world
    # block p of the send buffer: my rows of rank p's heads, [B, n, hn, D]
    send = x.reshape(B, n, world, hn, D).permute(2, 0, 1, 3, 4).contiguous().reshape(-1)
    recv = torch.empty(B * sum(seq_sizes) * hn * D, dtype=x.dtype, device=x.device)
    dist.all_to_all_single(recv, send, [B * m * hn * D for m in seq_sizes], [B * n * hn * D] * world, group=group)
    # block p of the receive buffer: rank p's rows of my heads, [B, n_p, hn, D]
    blocks = torch.split(recv, [B * m * hn * D for m in seq_sizes])
    return torch.cat([blk.view(B, m, hn, D) for blk, m in zip(blocks, seq_sizes)], dim=1)


def heads_to_seq(y, seq_sizes, group=None):
    """This rank's head shard [B, L, H/N, D] -> its sequence shard [B, n_rank, H, D] (one all-to-all)."""
    world, rank = _world(group), _rank(group)
    B, L, hn, D = y.shape
    if world == 1:
        return y.contiguous()
    if L != sum(seq_sizes) or len(seq_sizes) != world:
        raise ValueError("the head shard does not match seq_sizes")
    n = seq_sizes[rank]
    # block p of the send buffer: rank p's rows of my heads
    send = torch.cat([blk.reshape(-1) for blk in torch.split(y, seq_sizes, dim=1)])
    recv = torch.empty(B * n * hn * D * world, dtype=y.dtype, device=y.device)
    dist.all_to_all_single(recv, send, [B * n * hn * D] * world, [B * m * hn * D for m in seq_sizes], group=group)
    # block p of the receive buffer: my rows of rank p's heads, [B, n, hn, D]
    return recv.view(world, B, n, hn, D).permute(1, 2, 0, 3, 4).reshape(B, n, world * hn, D)


def forward_heads(q, k, v, h0, nh, T, S, K, r, G, global_pos=0, out=None):
    """Window attention of the heads [h0, h0 + nh) of [B, L, H, D] bf16 CUDA tensors (any strides the library
    accepts), written into the same heads of `out` (allocated like q when None); other heads of `out` are left as
    they are. One plan with H = nh and the tensors' own strides, on views that start at head h0."""
    from . import Plan
    B, L, H, D = q.shape
    if not 0 <= h0 < h0 + nh <= H:
        raise ValueError(f"head range [{h0}, {h0 + nh}) outside [0, {H})")
    if out is None:
        out = torch.empty_like(q)
    plan = Plan(T, S, K, r, G, B, nh, D, global_pos, strides=tuple(q.stride()[:3]))
    try:
        sel = slice(h0, h0 + nh)
        plan.forward(q[:, :, sel], k[:, :, sel], v[:, :, sel], out=out[:, :, sel])
    finally:
        plan.close()
    return out


def sharded_forward(q, k, v, T, S, K, r, G, global_pos=0, seq_sizes=None, group=None, attend=None):
    """Window attention of a sequence-sharded layer: q, k, v are this rank's [B, n_rank, H, D] sequence shards;
    returns this rank's [B, n_rank, H, D] shard of the output.

    q, k and v go to head shards (three all-to-alls), this rank's H/N heads are computed over the whole sequence,
    and the output comes back (one all-to-all). `attend(q, k, v)` computes the head shard; by default a plan of the
    library on the current CUDA device (``Plan.forward``). It is a parameter so that the exchange can be tested on
    ranks without a GPU with a stand-in that has the same shapes.
    """
    world = _world(group)
    L = T * S + G
    if seq_sizes is None:
        seq_sizes = even_seq_sizes(L, world)
    if sum(seq_sizes) != L:
        raise ValueError(f"seq_sizes sum to {sum(seq_sizes)}, not L = {L}")
    qh, kh, vh = (seq_to_heads(t, seq_sizes, group) for t in (q, k, v))
    if attend is None:
        from . import Plan
        B, _, hn, D = qh.shape
        plan = Plan(T, S, K, r, G, B, hn, D, global_pos)
        try:
            oh = plan.forward(qh, kh, vh)
        finally:
            plan.close()
    else:
        oh = attend(qh, kh, vh)
    return heads_to_seq(oh, seq_sizes, group)
