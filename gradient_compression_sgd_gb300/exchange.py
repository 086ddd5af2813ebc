"""The exchange step across ranks, one process per GPU.

"Deep Gradient Compression", Appendix A (synchronous distributed SGD) and
section 5: every node's sparse gradient reaches every other node, which sums
them.  "AdaComp", Proposed method: each learner receives the other learners'
compressed gradients and averages them.  With K learners spread over the W
ranks of a process group, rank r compresses learners [lo_r, hi_r) (a
contiguous, as-even-as-possible split, `learner_range`) and `exchange_average`
then

  1. all-gathers the per-learner entry counts;
  2. all-gathers the packed (index, value) lists, each cut to the largest
     count over all K learners (the counts bound every list, so the padding
     is never read);
  3. runs the K-way sparse average over the gathered lists in global learner
     order.

Every rank ends with the same dense average, and it is bit for bit the one a
single process holding all K learners computes: the average adds the lists
in learner order 0..K-1 whichever rank compressed them.  An all-gather of
lists is used rather than an all-reduce of sparse sums, whose density can
double at each reduction step (DGC, section 5).

"Communication Compression for Decentralized Training", DCD-PSGD step 3:
ring node i sends C(z_i) to its two neighbours, which add it to their copies
of x_i.  `RingPartition` places nodes [a, b) on rank r with copies of the two
boundary neighbours a-1 and b (mod n) beside them; `ring_iteration` steps
the own nodes, `ring_exchange` sends the packed C of the first and last own
node to the neighbouring ranks and receives theirs, and each received C is
added to its copy, which then holds the owner's exact fp32 result.  The
packed C holds every entry the owner's C(z) can change a copy by (on the GPU,
every kept entry: `GpuRing`).

Only torch.distributed calls (all_gather, isend/irecv) move data: with NCCL
on CUDA tensors and gloo on CPU tensors alike.  The compression and the
average themselves are the library's kernels, passed in by the caller.
"""
from __future__ import annotations


def learner_range(K: int, world: int, rank: int) -> tuple[int, int]:
    """Learners [lo, hi) of `rank` when K learners are split over `world`
    ranks: contiguous blocks, the first K % world ranks one larger."""
    if K < 1 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"learner_range: K={K}, world={world}, rank={rank}")
    base, extra = divmod(K, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def _group_size(group):
    import torch.distributed as dist
    return dist.get_world_size(group), dist.get_rank(group)


def gather_lists(lists, totals, K: int, group=None):
    """All ranks' messages in global learner order.

    lists: [K_r, cap, 2] int32 pair records of this rank's learners (in
    learner order); totals: [K_r] int64 entries per list.  Returns
    (lists [K, cap_pad, 2] int32, totals [K] int64) on the same device,
    cap_pad = max(1, the largest count over all learners)."""
    import torch
    import torch.distributed as dist
    world, rank = _group_size(group)
    lo, hi = learner_range(K, world, rank)
    k_loc = hi - lo
    if lists.shape[0] != k_loc or totals.numel() != k_loc:
        raise ValueError(f"gather_lists: rank {rank} holds learners [{lo}, {hi}) but got {lists.shape[0]} lists "
                         f"and {totals.numel()} counts")
    k_max = learner_range(K, world, 0)[1]  # rank 0 holds the largest share
    dev = lists.device
    # 1. the counts
    cnt = torch.zeros(k_max, dtype=torch.int64, device=dev)
    cnt[:k_loc] = totals.reshape(-1).to(torch.int64)
    cnts = [torch.empty_like(cnt) for _ in range(world)]
    dist.all_gather(cnts, cnt, group=group)
    per_rank = [learner_range(K, world, r)[1] - learner_range(K, world, r)[0] for r in range(world)]
    totals_all = torch.cat([cnts[r][:per_rank[r]] for r in range(world)])
    cap = lists.shape[1]
    cap_pad = max(1, int(totals_all.max().item()))
    if cap_pad > cap:
        raise ValueError(f"gather_lists: a learner's count {cap_pad} exceeds the list capacity {cap}")
    # 2. the lists, cut to the longest message
    send = torch.zeros((k_max, cap_pad, 2), dtype=torch.int32, device=dev)
    send[:k_loc] = lists[:, :cap_pad]
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    lists_all = torch.cat([recv[r][:per_rank[r]] for r in range(world)])
    return lists_all.contiguous(), totals_all.contiguous()


def exchange_average(lists, totals, K: int, n: int, out, average=None, group=None):
    """The dense K-way average of every rank's messages, on every rank.

    `average(lists, counts, n, out)` defaults to the library's
    sparse_average; out: [n] fp32 on the lists' device.  Returns the gathered
    (lists, totals)."""
    if average is None:
        from . import sparse_average as average
    lists_all, totals_all = gather_lists(lists, totals, K, group)
    average(lists_all, totals_all, n, out)
    return lists_all, totals_all


# ------------------------------------------------------------ DCD-PSGD ring

class RingPartition:
    """Nodes [a, b) of a ring of n on rank r of `world`, with the layout of
    the rank's local rows: row 0 is a copy of node a-1, rows 1..b-a the own
    nodes a..b-1, row b-a+1 a copy of node b (indices mod n).  With world = 1
    there are no copies: the rows are the whole ring and it wraps locally."""

    def __init__(self, n: int, world: int, rank: int):
        if world > 1 and n < world:
            raise ValueError(f"RingPartition: {n} nodes cannot be spread over {world} ranks")
        self.n, self.world, self.rank = n, world, rank
        self.a, self.b = learner_range(n, world, rank)
        self.left_rank = (rank - 1) % world
        self.right_rank = (rank + 1) % world

    @property
    def own(self) -> int:
        return self.b - self.a

    @property
    def rows(self) -> int:
        """Local rows: the own nodes plus the two neighbour copies (world > 1)."""
        return self.own + (2 if self.world > 1 else 0)

    def row_nodes(self) -> list[int]:
        """Global node index of every local row."""
        if self.world == 1:
            return list(range(self.n))
        return [(self.a - 1) % self.n, *range(self.a, self.b), self.b % self.n]


# tags: which copy on the receiving rank a message is for
_TAG_FOR_LEFT_COPY, _TAG_FOR_RIGHT_COPY = 11, 12


def ring_exchange(part: RingPartition, first_c, last_c, group=None):
    """Sends the packed C of the first own node (node a) to the left rank,
    whose right copy it is, and of the last own node (b-1) to the right rank,
    whose left copy it is; receives C of nodes a-1 and b.

    first_c, last_c: [m, 2] int32 pair records (index, value bits) with
    unique indices, in any order.  Returns (C for the left copy, C for the right copy) as [m', 2]
    int32 pair tensors.  Counts go first (one int64 each way), then the
    pairs."""
    import torch
    import torch.distributed as dist
    if part.world == 1:
        raise ValueError("ring_exchange: a single rank holds the whole ring")
    left = dist.get_global_rank(group, part.left_rank) if group is not None else part.left_rank
    right = dist.get_global_rank(group, part.right_rank) if group is not None else part.right_rank
    dev = first_c.device

    def swap(send_left, send_right):
        r_left = torch.empty_like(send_left)
        r_right = torch.empty_like(send_right)
        ops = [dist.P2POp(dist.isend, send_left, left, group, _TAG_FOR_RIGHT_COPY),
               dist.P2POp(dist.isend, send_right, right, group, _TAG_FOR_LEFT_COPY),
               dist.P2POp(dist.irecv, r_left, left, group, _TAG_FOR_LEFT_COPY),
               dist.P2POp(dist.irecv, r_right, right, group, _TAG_FOR_RIGHT_COPY)]
        for req in dist.batch_isend_irecv(ops):
            req.wait()
        return r_left, r_right

    n_first = torch.tensor([first_c.shape[0]], dtype=torch.int64, device=dev)
    n_last = torch.tensor([last_c.shape[0]], dtype=torch.int64, device=dev)
    got_left_n, got_right_n = swap(n_first, n_last)
    cl, cr = int(got_left_n.item()), int(got_right_n.item())
    # pad to at least one record: a zero-length message is not sent
    pad = lambda c: c if c.shape[0] > 0 else torch.zeros((1, 2), dtype=torch.int32, device=dev)
    r_left = torch.empty((max(cl, 1), 2), dtype=torch.int32, device=dev)
    r_right = torch.empty((max(cr, 1), 2), dtype=torch.int32, device=dev)
    s_first, s_last = pad(first_c.contiguous()), pad(last_c.contiguous())
    ops = [dist.P2POp(dist.isend, s_first, left, group, _TAG_FOR_RIGHT_COPY),
           dist.P2POp(dist.isend, s_last, right, group, _TAG_FOR_LEFT_COPY),
           dist.P2POp(dist.irecv, r_left, left, group, _TAG_FOR_LEFT_COPY),
           dist.P2POp(dist.irecv, r_right, right, group, _TAG_FOR_RIGHT_COPY)]
    for req in dist.batch_isend_irecv(ops):
        req.wait()
    return r_left[:cl], r_right[:cr]


def ring_iteration(part: RingPartition, xrows, g_own, t: int, step, copy_add, group=None):
    """One DCD-PSGD iteration across ranks on this rank's rows.

    step(xrows, g_own, t) updates the own rows and returns the packed C of the
    first and the last own node ([m, 2] int32 pairs each); the two lists go
    to the neighbouring ranks and theirs come back; copy_add(row, pairs) adds
    a received C to a copy row.  With world = 1 the rows are the whole ring
    and only step runs."""
    first, last = step(xrows, g_own, t)
    if part.world == 1:
        return
    got_left, got_right = ring_exchange(part, first, last, group)
    copy_add(xrows[0], got_left)
    copy_add(xrows[-1], got_right)


class GpuRing:
    """The library's kernels as ring_iteration's step and copy_add, for one
    rank's rows on its GPU: dcd_step_rows (lists sized to d, so no kept entry
    is ever dropped) and dcd_copy_add.  The first copy update of a copy row
    also adds +0 to every entry (dcd_copy_add's zero pass), which makes a
    starting model with -0 entries agree with its owner bit for bit."""

    def __init__(self, part: RingPartition, d: int, w_ring, gamma: float, keep_p: float, seed: int, device):
        import torch
        self.part, self.d = part, d
        self.w, self.gamma, self.p, self.seed = w_ring, gamma, keep_p, seed
        self.first = torch.empty((max(d, 1), 2), dtype=torch.int32, device=device)
        self.last = torch.empty((max(d, 1), 2), dtype=torch.int32, device=device)
        self.counts = torch.zeros(2, dtype=torch.int64, device=device)
        self.recv_count = torch.zeros(1, dtype=torch.int64, device=device)
        self.zero_pass_done = set()

    def step(self, xrows, g_own, t):
        from . import dcd_step_rows
        dcd_step_rows(xrows, g_own, self.w, self.gamma, self.p, self.seed, t, self.part.a, self.first, self.last,
                      self.counts)
        nf, nl = (int(c) for c in self.counts.tolist())  # the message sizes are needed on the host to send
        return self.first[:nf], self.last[:nl]

    def copy_add(self, row, pairs):
        from . import dcd_copy_add
        key = row.data_ptr()
        self.recv_count.fill_(pairs.shape[0])
        dcd_copy_add(row, pairs.contiguous(), self.recv_count, zero_pass=key not in self.zero_pass_done)
        self.zero_pass_done.add(key)
