"""One rank of a multi-GPU TSP layer: the host-side schedule of its compute
steps and of the exchanges between ranks.

Tensor and Sequence Parallelism folds the tensor- and sequence-parallel axes
into one axis of D ranks: rank r holds 1/D of the tokens (zigzag chunks r and
2D-1-r of every sequence) and 1/D of the weights (ai-trends.today, "Zyphra
Introduces Tensor and Sequence Parallelism (TSP)", section "How to Fold a
Book").  One layer forward on rank r:

* attention: for every shard s, its owner broadcasts the packed {W_Q, W_K,
  W_V, W_O} shard; every rank projects its own tokens, the local K/V are
  all-gathered (and put back into natural order), causal attention runs for
  the rank's queries, and the W_O partial product is accumulated locally;
* gated MLP: a ring over the gate/up/down shards -- at step t rank r holds
  shard (r - t) mod D, starting from its own, and passes it to rank r + 1 --
  accumulating partial outputs, with no output all-reduce.

Weight transfers are hidden behind the GEMMs ("The Practicality of
Trade-offs"): the broadcast of shard s+1 and the ring hop of the next MLP
shard are in flight while the current shard computes (double-buffered
receive slots).  The K/V all-gather is a true dependency of the attention.

The compute steps are the per-rank C ABI calls (``tsp_rank_qkv``,
``tsp_rank_attention``, ``tsp_rank_mlp``) through :class:`RankLayer`; the
exchanges go through a communicator:

* :class:`DistComm` -- ``torch.distributed`` (NCCL between GPUs, gloo on
  CPU), one process per rank.  Every wait is bounded; a rank whose wait runs
  out records that it gave up in the process group's store and raises
  ``TspError(TSP_ERR_TIMEOUT)``; the other ranks see the record before their
  next exchange and give up too, instead of waiting on a peer that left.
* :class:`LocalComm` -- D virtual ranks in one process on one GPU, each a
  host thread with its own CUDA stream; an exchange is a host rendezvous plus
  device copies ordered by CUDA events (no kernel ever waits on another).

Every buffer handed to a kernel is local to the rank: a shard received from
another rank is first copied into a local receive slot.
"""

from __future__ import annotations

import datetime
import threading
from typing import Callable, Optional

from .tsp import TSP_ERR_TIMEOUT, TspError

ABORT_KEY = "tsp_rank/gave_up"


# ---- the schedule ------------------------------------------------------------------


def layer_fwd(comm, compute, x_local, attn_own, mlp_own):
    """Rank ``comm.rank``'s part of one TSP layer forward.

    ``x_local``: the rank's zigzag token rows [batch*2C][h]; ``attn_own`` /
    ``mlp_own``: the attention and MLP weight shards the rank owns (shard
    index = rank).  ``compute`` provides the per-rank compute steps and the
    receive buffers (``attn_recv``, ``mlp_recv``: two slots each, ``kv_all``,
    ``h``, ``y``).  Returns ``compute.y``, the rank's rows of the layer output.
    """
    D, r = comm.world_size, comm.rank

    def attn_slot(s):
        return attn_own if s == r else compute.attn_recv[s % 2]

    pending = comm.broadcast(attn_slot(0), 0)
    for s in range(D):
        pending.wait()
        cur = attn_slot(s)
        if s + 1 < D:  # the next shard travels while this one computes
            pending = comm.broadcast(attn_slot(s + 1), s + 1)
        kv = compute.project(x_local, cur)
        comm.all_gather(compute.kv_all, kv).wait()
        compute.attend(cur, x_local if s == 0 else compute.h)
    cur = mlp_own
    for t in range(D):
        nxt = None
        if t + 1 < D:  # pass the current shard on and receive the next during this step
            nxt = compute.mlp_recv[t % 2]
            pending = comm.ring_shift(cur, nxt)
        compute.mlp(cur, compute.h if t == 0 else compute.y)
        if nxt is not None:
            pending.wait()
            cur = nxt
    return compute.y


# ---- the rank's compute steps on its GPU ---------------------------------------------


class RankLayer:
    """Buffers and per-rank C ABI calls of one rank (its local rows, the
    receive slots for shards from other ranks, and the workspaces)."""

    def __init__(self, plan, rank: int, batch: int, device=None, stream=None):
        import torch

        from . import tsp

        self.tsp, self.plan, self.rank, self.batch = tsp, plan, rank, batch
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.stream = stream
        D, h = plan.D, plan.hidden
        C = plan.seq // (2 * D)
        L = batch * 2 * C
        hs, ks = h // D, plan.kv_hidden // D
        dt, dev = plan.torch_dtype, self.device
        self.rows = L
        self.q = torch.empty(L, hs, dtype=dt, device=dev)
        self.kv = torch.empty(L, 2 * ks, dtype=dt, device=dev)
        self.kv_all = torch.empty(D, L, 2 * ks, dtype=dt, device=dev)
        self.h = torch.empty(L, h, dtype=dt, device=dev)
        self.y = torch.empty(L, h, dtype=dt, device=dev)
        na = tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_ATTENTION)
        nm = tsp.tsp_rank_shard_bytes(plan, tsp.TSP_SHARD_MLP)
        self.attn_recv = [torch.empty(na, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.mlp_recv = [torch.empty(nm, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.attn_ws = tsp.workspace(plan, batch, tsp.TSP_OP_RANK_ATTENTION, dev)
        self.mlp_ws = tsp.workspace(plan, batch, tsp.TSP_OP_RANK_MLP, dev)

    def own_shards(self, packed):
        """The attention and MLP shards this rank owns, cut from whole packed weights."""
        import torch

        t = self.tsp
        a = torch.empty(t.tsp_rank_shard_bytes(self.plan, t.TSP_SHARD_ATTENTION), dtype=torch.uint8,
                        device=self.device)
        m = torch.empty(t.tsp_rank_shard_bytes(self.plan, t.TSP_SHARD_MLP), dtype=torch.uint8, device=self.device)
        t.tsp_rank_extract_shard(self.plan, packed, self.rank, t.TSP_SHARD_ATTENTION, a, self.stream)
        t.tsp_rank_extract_shard(self.plan, packed, self.rank, t.TSP_SHARD_MLP, m, self.stream)
        return a, m

    def project(self, x_local, attn_shard):
        self.tsp.tsp_rank_qkv(self.plan, self.batch, x_local, attn_shard, self.q, self.kv, self.stream)
        return self.kv

    def attend(self, attn_shard, resid):
        self.tsp.tsp_rank_attention(self.plan, self.rank, self.batch, self.q, self.kv_all, attn_shard, resid, self.h,
                                    self.attn_ws, self.stream)

    def mlp(self, mlp_shard, resid):
        self.tsp.tsp_rank_mlp(self.plan, self.batch, self.h, mlp_shard, resid, self.y, self.mlp_ws, self.stream)


# ---- exchanges over torch.distributed -------------------------------------------------


class _DistWork:
    def __init__(self, comm, works, what):
        self.comm, self.works, self.what = comm, works, what

    def wait(self):
        for w in self.works:
            try:
                if self.comm.timeout is not None:
                    w.wait(timeout=self.comm.timeout)
                else:
                    w.wait()
            except RuntimeError as e:
                self.comm.give_up(self.what, str(e))
        return self


class DistComm:
    """The exchanges of the TSP schedule over a ``torch.distributed`` group.

    ``timeout_s``: bound on every wait (None: the group's own timeout).
    ``store``: where a rank that gave up says so (default: the default
    group's store); every exchange first checks it.  ``drop_send``: host-side
    fault injection for tests -- called with the ring step index, a True
    return makes this rank skip that step's send (its receive still runs).
    """

    def __init__(self, group=None, timeout_s: Optional[float] = None, store=None,
                 drop_send: Optional[Callable[[int], bool]] = None):
        import torch.distributed as dist

        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world_size = dist.get_world_size(group)
        self.timeout = datetime.timedelta(seconds=timeout_s) if timeout_s is not None else None
        if store is None:
            from torch.distributed import distributed_c10d

            store = distributed_c10d._get_default_store()
        self.store = store
        self.drop_send = drop_send
        self.ring_step = 0

    def _global(self, r):
        return self.dist.get_global_rank(self.group, r) if self.group is not None else r

    def check_peers(self, what: str):
        """Raises TspError(TSP_ERR_TIMEOUT) if another rank has given up (or
        the store that would say so cannot be reached)."""
        try:
            gone = self.store.check([ABORT_KEY])
            who = self.store.get(ABORT_KEY).decode(errors="replace") if gone else None
        except RuntimeError as e:  # the store's host is gone: so is the group
            raise TspError(TSP_ERR_TIMEOUT, what, f"store unreachable ({str(e).splitlines()[0][:120]})") from e
        if gone:
            raise TspError(TSP_ERR_TIMEOUT, what, f"rank {who} gave up; not starting the exchange")

    def give_up(self, what: str, detail: str):
        try:
            self.store.set(ABORT_KEY, str(self.rank))
        except RuntimeError:
            pass  # the others then find out from their own bounded waits
        raise TspError(TSP_ERR_TIMEOUT, what, f"rank {self.rank}: wait gave up ({detail.splitlines()[0][:160]})")

    def broadcast(self, buf, src: int):
        what = f"broadcast of attention shard {src}"
        self.check_peers(what)
        w = self.dist.broadcast(buf, src=self._global(src), group=self.group, async_op=True)
        return _DistWork(self, [w], what)

    def all_gather(self, out, inp):
        what = "K/V all-gather"
        self.check_peers(what)
        flat = out.view(-1, *inp.shape[1:])  # [D][rows][cols] as the ranks' rows one after another
        w = self.dist.all_gather_into_tensor(flat, inp, group=self.group, async_op=True)
        return _DistWork(self, [w], what)

    def ring_shift(self, send, recv):
        step = self.ring_step
        self.ring_step += 1
        what = f"MLP ring step {step + 1}"
        self.check_peers(what)
        D, r = self.world_size, self.rank
        # Each hop carries its step as the message tag, so a lost hop can never
        # be matched by the next one (which would hand the receiver the wrong shard).
        tag = step + 1
        ops = [self.dist.P2POp(self.dist.irecv, recv, self._global((r - 1) % D), self.group, tag)]
        if not (self.drop_send is not None and self.drop_send(step)):
            ops.insert(0, self.dist.P2POp(self.dist.isend, send, self._global((r + 1) % D), self.group, tag))
        return _DistWork(self, self.dist.batch_isend_irecv(ops), what)


# ---- D virtual ranks in one process (one GPU) --------------------------------------------


class _Rendezvous:
    """Shared state of the virtual ranks: a barrier and one slot per rank."""

    def __init__(self, D: int, timeout_s: float):
        self.D = D
        self.barrier = threading.Barrier(D, timeout=timeout_s)
        self.slot = [None] * D
        self.done = [None] * D


class _Done:
    def wait(self):
        return self


class LocalComm:
    """The exchanges of the TSP schedule between D virtual ranks, each a host
    thread with its own CUDA stream on the same GPU.

    An exchange: every rank posts (buffer, event recorded on its stream) and
    meets the others at a barrier; each receiver's stream waits on the
    sender's event and copies the data; the copies' events are posted, and
    after a second barrier the sender's stream waits on them, so the sender
    reuses its buffer only once the copies are done.  All waiting is
    host-side or stream-ordered.
    """

    def __init__(self, rdv: _Rendezvous, rank: int, stream):
        self.rdv, self.rank, self.world_size, self.stream = rdv, rank, rdv.D, stream

    def _event(self):
        import torch

        e = torch.cuda.Event()
        e.record(self.stream)
        return e

    def _exchange(self, post, copy, readers_of_mine):
        import torch

        rdv, r = self.rdv, self.rank
        rdv.slot[r] = (post, self._event())
        rdv.barrier.wait()
        with torch.cuda.stream(self.stream):
            copy()
        rdv.done[r] = self._event()
        rdv.barrier.wait()
        # My posted buffer is free once every reader has copied it.  (A rank
        # reposts its slot and event only after the next exchange's first
        # barrier, which every rank reaches after reading these.)
        for q in readers_of_mine:
            self.stream.wait_event(rdv.done[q])
        return _Done()

    def broadcast(self, buf, src: int):
        rdv, r = self.rdv, self.rank

        def copy():
            if r != src:
                sbuf, ev = rdv.slot[src]
                self.stream.wait_event(ev)
                buf.copy_(sbuf, non_blocking=True)

        readers = [q for q in range(self.world_size) if q != src] if r == src else []
        return self._exchange(buf, copy, readers)

    def all_gather(self, out, inp):
        rdv = self.rdv

        def copy():
            for q in range(self.world_size):
                sbuf, ev = rdv.slot[q]
                self.stream.wait_event(ev)
                out[q].copy_(sbuf, non_blocking=True)

        return self._exchange(inp, copy, list(range(self.world_size)))

    def ring_shift(self, send, recv):
        rdv, r, D = self.rdv, self.rank, self.world_size

        def copy():
            sbuf, ev = rdv.slot[(r - 1) % D]
            self.stream.wait_event(ev)
            recv.copy_(sbuf, non_blocking=True)

        return self._exchange(send, copy, [(r + 1) % D])


def run_local_ranks(D: int, body, timeout_s: float = 600.0):
    """Runs ``body(rank, comm)`` for ranks 0..D-1 as D host threads of this
    process (one GPU, one CUDA stream per rank) and returns their results in
    rank order.  An exception in any rank breaks the barrier for the others
    and is re-raised here."""
    import torch

    rdv = _Rendezvous(D, timeout_s)
    dev = torch.cuda.current_device()
    results, errors = [None] * D, [None] * D

    def run(rank):
        torch.cuda.set_device(dev)
        stream = torch.cuda.Stream(device=dev)
        try:
            results[rank] = body(rank, LocalComm(rdv, rank, stream))
            stream.synchronize()
        except BaseException as e:  # noqa: BLE001 -- handed to the caller below
            errors[rank] = e
            rdv.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,), name=f"tsp-rank-{r}") for r in range(D)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for e in errors:
        if e is not None and not isinstance(e, threading.BrokenBarrierError):
            raise e
    for e in errors:
        if e is not None:
            raise e
    return results
