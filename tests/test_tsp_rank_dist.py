"""The multi-GPU TSP schedule (folded_tensor_sequence_gb300.tsp_rank) run by
real ranks: D processes over torch.distributed's gloo backend on the CPU,
each computing its steps in fp64 with the oracle's definitions
(tests/rank_oracle.py), exchanging shards and K/V through DistComm.

Checked on every rank:
* after each broadcast the attention shard it computes with is, bit for bit,
  the owner's shard in the tsp_rank_* layout (oracle ``attention_shard``);
* after each all-gather, rank q's K/V rows put at the oracle's zigzag
  positions of rank q give exactly the full K, V of the shard's heads
  (x Wk, x Wv of the unsharded layer);
* at MLP ring step t it holds shard (r - t) mod D, bit for bit (oracle
  ``mlp_shard``) -- the ring starts at the rank's own shard;
* its output rows equal the oracle's sharded and unsharded layers at its
  zigzag positions (fp64, 1e-12).

And the failure path: one rank drops its send of an MLP ring hop; the rank
that waits for it gives up after its bounded wait with TSP_ERR_TIMEOUT,
records that in the store, and every rank returns (none waits forever).
"""
import datetime
import multiprocessing as mp
import os
import socket
import time
import traceback

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CASES = {
    # D, batch, seq, hidden, heads, kv_heads, ffn (ffn/D a multiple of 128: whole gate/up blocks per shard)
    "D2_gqa": (2, 2, 16, 64, 4, 2, 256),
    "D4_mha": (4, 1, 32, 64, 4, 4, 512),
}


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, case, mode, q):
    import sys

    sys.path[:0] = [ROOT, HERE]
    try:
        import torch
        import torch.distributed as dist

        from folded_tensor_sequence_gb300 import synth
        from folded_tensor_sequence_gb300.configs import LayerConfig
        from folded_tensor_sequence_gb300.tsp import TSP_ERR_TIMEOUT, TspError
        from folded_tensor_sequence_gb300.tsp_rank import ABORT_KEY, DistComm, layer_fwd
        from oracle import tsp_oracle as O
        from rank_oracle import OracleRankCompute, pack_attention_shard, pack_mlp_shard

        D, B, S, h, H, Hk, F = CASES[case]
        assert D == world
        # the parent process hosts the store, so it outlives any rank that leaves early
        store = dist.TCPStore("127.0.0.1", port, is_master=False, timeout=datetime.timedelta(seconds=60))
        dist.init_process_group("gloo", store=store, rank=rank, world_size=world,
                                timeout=datetime.timedelta(seconds=60))
        cfg = LayerConfig(case, D=D, batch=B, seq=S, hidden=h, heads=H, head_dim=h // H, ffn=F, dtype="f32",
                          kv_heads=Hk)
        inp = synth.layer_inputs(cfg, seed=7)  # every rank draws the same seeded inputs
        w = {k: inp[k] for k in ("Wq", "Wk", "Wv", "Wo", "Wg", "Wu", "Wd")}
        xz = O.zigzag_permute(inp["x"], D)  # [D, B, 2C, h]: this rank keeps xz[rank] only
        x_local = torch.from_numpy(np.ascontiguousarray(xz[rank].reshape(-1, h)))
        attn_own = torch.from_numpy(pack_attention_shard(w, rank, D))
        mlp_own = torch.from_numpy(pack_mlp_shard(w, rank, D))
        comp = OracleRankCompute(rank, D, B, S, h, H, Hk, F)
        if mode == "drop":
            # rank 0 skips its send of the first ring hop; rank 1 waits for it
            comm = DistComm(timeout_s=1.5, store=store, drop_send=(lambda step: rank == 0 and step == 0))
            t0 = time.time()
            status, msg, err = 0, "", None
            try:
                y = layer_fwd(comm, comp, x_local, attn_own, mlp_own).numpy()
                # a rank that finished got every hop it needed: its rows must be right
                pos = O.zigzag_positions(S, D)
                ref = O.layer_fwd(inp["x"], w, H)["Y"]
                err = max(float(np.max(np.abs(y.reshape(B, -1, h)[b] - ref[b, pos[rank]]))) for b in range(B))
            except TspError as e:
                status, msg = e.status, str(e)
            q.put((rank, {"status": status, "msg": msg, "secs": time.time() - t0, "err": err,
                          "timeout_code": TSP_ERR_TIMEOUT, "abort": store.check([ABORT_KEY])}))
            _flush_and_exit(q, 0)  # a rank that gave up may still have a receive posted: leave without teardown
        comm = DistComm(timeout_s=30.0, store=store)
        y = layer_fwd(comm, comp, x_local, attn_own, mlp_own).numpy().copy()
        # what travelled
        pos = O.zigzag_positions(S, D)
        attn_ok = all(np.array_equal(comp.seen_attn[s].numpy(), pack_attention_shard(w, s, D)) for s in range(D))
        mlp_ok = all(np.array_equal(comp.seen_mlp[t].numpy(), pack_mlp_shard(w, (rank - t) % D, D))
                     for t in range(D))
        ks = Hk * (h // H) // D
        kv_err = 0.0
        x = inp["x"]
        for s in range(D):
            kv_all = comp.seen_kv_all[s].numpy()
            _, Wk_s, Wv_s, _ = O.attention_shard(w, s, D)
            for b in range(B):
                Kn = np.zeros((S, ks))
                Vn = np.zeros((S, ks))
                for qr in range(D):
                    rows = kv_all[qr, b * 2 * (S // (2 * D)):(b + 1) * 2 * (S // (2 * D))]
                    Kn[pos[qr]] = rows[:, :ks]
                    Vn[pos[qr]] = rows[:, ks:]
                kv_err = max(kv_err, float(np.max(np.abs(Kn - x[b] @ Wk_s))), float(np.max(np.abs(Vn - x[b] @ Wv_s))))
        ref_sh = O.tsp_layer_fwd_sharded(x, w, H, D)["Y"]
        ref = O.layer_fwd(x, w, H)["Y"]
        mine = y.reshape(B, -1, h)
        e_sh = max(float(np.max(np.abs(mine[b] - ref_sh[b, pos[rank]]))) for b in range(B)) / float(np.max(np.abs(ref)))
        e_un = max(float(np.max(np.abs(mine[b] - ref[b, pos[rank]]))) for b in range(B)) / float(np.max(np.abs(ref)))
        q.put((rank, {"attn_ok": attn_ok, "mlp_ok": mlp_ok, "kv_err": kv_err, "err_sharded": e_sh,
                      "err_plain": e_un, "n_attn": len(comp.seen_attn), "n_mlp": len(comp.seen_mlp)}))
        dist.destroy_process_group()
    except BaseException:  # noqa: BLE001 -- reported to the parent
        q.put((rank, {"error": traceback.format_exc()}))
        _flush_and_exit(q, 1)


def _flush_and_exit(q, code):
    q.close()
    q.join_thread()  # the queue's feeder thread has handed the result over
    os._exit(code)


def _run(world, case, mode, limit_s=120):
    import torch.distributed as dist

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    server = dist.TCPStore("127.0.0.1", port, is_master=True, wait_for_workers=False,  # noqa: F841 -- kept alive
                           timeout=datetime.timedelta(seconds=60))
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    deadline = time.time() + limit_s
    while len(out) < world and time.time() < deadline:
        try:
            r, res = q.get(timeout=max(0.1, deadline - time.time()))
            out[r] = res
        except Exception:  # noqa: BLE001 -- queue.Empty
            break
    for p in procs:
        p.join(timeout=max(1.0, deadline - time.time()))
    for p in procs:
        if p.is_alive():  # only our own children, by handle
            p.kill()
            p.join()
    return out, [p.exitcode for p in procs]


@pytest.mark.parametrize("case", sorted(CASES))
def test_schedule_across_ranks(case):
    world = CASES[case][0]
    out, codes = _run(world, case, "run")
    assert len(out) == world, (out, codes)
    for r in range(world):
        res = out[r]
        assert "error" not in res, res.get("error")
        assert res["n_attn"] == world and res["n_mlp"] == world
        assert res["attn_ok"], f"rank {r}: a broadcast attention shard differs from its owner's"
        assert res["mlp_ok"], f"rank {r}: the MLP ring handed a wrong shard"
        assert res["kv_err"] <= 1e-12, f"rank {r}: gathered K/V off by {res['kv_err']}"
        assert res["err_sharded"] <= 1e-12, res
        assert res["err_plain"] <= 1e-12, res
    assert codes == [0] * world


def test_dropped_ring_message_times_out_on_every_rank():
    world = 4
    out, codes = _run(world, "D4_mha", "drop", limit_s=90)
    assert len(out) == world, (out, codes)
    timeout_code = out[0]["timeout_code"]
    # the rank waiting for the dropped hop gives up after its bounded wait
    assert out[1]["status"] == timeout_code, out[1]
    assert "gave up" in out[1]["msg"]
    for r in range(world):
        assert out[r]["status"] in (0, timeout_code), out[r]
        assert out[r]["secs"] < 30, f"rank {r} took {out[r]['secs']:.1f} s"
    # rank 2 then waits for rank 1's next hop, which never comes, and rank 3 for rank 2's
    for r in (2, 3):
        assert out[r]["status"] == timeout_code, out[r]
    # the one that gave up first says so in the store
    assert out[1]["abort"]
    # rank 0 receives from rank 3, which sent every hop before waiting: if it finished, it is right
    for r in range(world):
        if out[r]["status"] == 0:
            assert out[r]["err"] <= 1e-12, out[r]
    assert codes == [0] * world


class _DeadStore:
    """A store whose host is gone: every call fails as a lost connection does."""

    def check(self, keys):
        raise RuntimeError("Connection reset by peer")

    def get(self, key):
        raise RuntimeError("Connection reset by peer")

    def set(self, key, value):
        raise RuntimeError("Broken pipe")


def test_unreachable_store_reads_as_a_timeout():
    from folded_tensor_sequence_gb300.tsp import TSP_ERR_TIMEOUT, TspError
    from folded_tensor_sequence_gb300.tsp_rank import DistComm

    comm = DistComm.__new__(DistComm)  # no process group needed for the store paths
    comm.rank, comm.store = 3, _DeadStore()
    for call in (lambda: comm.check_peers("K/V all-gather"), lambda: comm.give_up("MLP ring step 2", "timed out")):
        try:
            call()
        except TspError as e:
            assert e.status == TSP_ERR_TIMEOUT
        else:
            raise AssertionError("no error raised")
