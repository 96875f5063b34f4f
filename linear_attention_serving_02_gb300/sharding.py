"""Head sharding across ranks (tensor parallelism as the model is deployed, 'Kimi K3
attention deep dive', §6.1: the KDA state is split by head).

Every (sequence, head) unit of KDA is independent, so a rank that owns a contiguous block
of heads runs prefill and decode on its block alone; no collective is needed on the data
path. These helpers are host logic only: they pick a rank's heads and slice the head axis
of the inputs and states, which every entry point takes as [..., H, ...].
"""

HEAD_AXIS = {
    # name: the axis of H in that tensor
    "q": -2, "k": -2, "v": -2, "z": -2,   # [..., H, 128]
    "b": -1,                               # [..., H]
    "A": 0,                                # [H]
    "S0": 1, "state": 1,                   # [N, H, 128, 128]
}


def head_range(num_heads, rank, world):
    """[h0, h1): the contiguous block of heads rank `rank` of `world` owns. Blocks differ in
    size by at most one head; with fewer heads than ranks some blocks are empty."""
    if world <= 0 or not 0 <= rank < world or num_heads < 0:
        raise ValueError("need 0 <= rank < world and num_heads >= 0")
    base, extra = divmod(num_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def shard_heads(tensors, rank, world, num_heads):
    """The rank's slice of every tensor in `tensors` (a dict keyed as HEAD_AXIS; None
    values and names without a head axis pass through unchanged)."""
    h0, h1 = head_range(num_heads, rank, world)
    out = {}
    for name, t in tensors.items():
        ax = HEAD_AXIS.get(name)
        if t is None or ax is None:
            out[name] = t
            continue
        ax = ax % t.dim()
        if t.shape[ax] != num_heads:
            raise ValueError("%s has %d entries on its head axis, expected %d" % (name, t.shape[ax], num_heads))
        out[name] = t.narrow(ax, h0, h1 - h0).contiguous()
    return out
