"""Sequence-sharded prefill (linear_attention_hybrid_fwd_b300.sharded) on CPU, gloo.

Each rank holds one contiguous segment of the same sequences (uneven lengths); the
per-rank operations (prefill, state-only pass, ordered state sum) are fp64 oracle
stand-ins for the GPU kernels, so what is checked is the exchange: the all-gather of
segment states and the prefix each rank continues from.  The concatenated outputs
must equal the oracle run on the whole sequence, and the last rank's state the whole
sequence's final state, both to fp64 rounding.
"""
import os
import socket

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SEGMENTS = {2: [37, 50], 3: [37, 50, 13]}
B, H, D = 2, 2, 8


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(total):
    rng = np.random.default_rng(11)
    return [rng.standard_normal((B, total, H, D)) * 0.5 for _ in range(4)]


def _worker(rank, world, port, q_out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    import oracle
    from linear_attention_hybrid_fwd_b300.sharded import sharded_prefill
    dist.init_process_group("gloo", rank=rank, world_size=world)

    from oracle.state_pass import state_pass

    def prefill(q, k, v, g, kv_state_in=None, eps=1e-6):
        out, _, S = oracle.prefill(q.numpy(), k.numpy(), v.numpy(), g.numpy(),
                                   S0=None if kv_state_in is None else kv_state_in.numpy(),
                                   eps=eps)
        return torch.from_numpy(out), torch.from_numpy(S)

    def state(k, v):
        return torch.from_numpy(state_pass(k, v))

    def state_sum(parts, base=None):
        acc = torch.zeros_like(parts[0]) if base is None else base.clone()
        for p in parts:  # in rank order, as the library adds them
            acc = acc + p
        return acc

    ops = {"prefill": prefill, "state_pass": state, "state_sum": state_sum}

    seg = SEGMENTS[world]
    lo = sum(seg[:rank])
    q, k, v, g = (torch.from_numpy(np.ascontiguousarray(t[:, lo:lo + seg[rank]]))
                  for t in _inputs(sum(seg)))
    out, S = sharded_prefill(q, k, v, g, ops=ops)
    q_out.put((rank, out.numpy(), S.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_prefill_matches_whole_sequence(world, oracle_mod):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q_out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q_out.get(timeout=120) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    q, k, v, g = _inputs(sum(SEGMENTS[world]))
    ref_out, _, ref_S = oracle_mod.prefill(q, k, v, g)
    got = np.concatenate([r[1] for r in res], axis=1)
    np.testing.assert_allclose(got, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(res[-1][2], ref_S, rtol=1e-11, atol=1e-12)
    # an inner rank ends at the state of the sequence up to its segment's end
    n0 = SEGMENTS[world][0]
    _, _, S0 = oracle_mod.prefill(q[:, :n0], k[:, :n0], v[:, :n0], g[:, :n0])
    np.testing.assert_allclose(res[0][2], S0, rtol=1e-12, atol=1e-12)
