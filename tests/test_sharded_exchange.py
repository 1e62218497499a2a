"""The vocabulary-sharded step's exchange on CPU (gloo, world size 2).

A vocabulary-parallel LM head leaves each rank one shard of every logits
row; each rank reduces its shard to a (max, sum, argmax) triple per masked
position (12 bytes), the ranks all-gather the triples, and every rank merges
them in shard order and runs S3-S6.  Here the ranks are processes on the
CPU and the per-rank reduction is the oracle's; the test checks that the
gathered, merged result equals the unsharded step.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CFG = dict(B=3, L=8, V=301, O=6.0)
BOUNDS = [0, 152, 301]          # rank 0: [0, 152), rank 1: [152, 301)


def _case():
    import synth
    cfg = synth.StepConfig("xch", CFG["B"], CFG["L"], CFG["V"], CFG["O"], "fraction", (0.5, 0.8))
    inp = synth.make_step_state(cfg, 9)
    rows = np.flatnonzero(inp.masked.reshape(-1))
    logits = np.full((cfg.B * cfg.L, cfg.row_stride), synth.POISON_BITS, dtype=np.uint16)
    synth.fill_logits_rows(logits, cfg.V, rows, synth.step_row_keys(inp, rows), cfg.offset_max, cfg.mask_id)
    return cfg, inp, rows, logits


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg, inp, rows, logits = _case()
    lo, hi = BOUNDS[rank], BOUNDS[rank + 1]
    mine = torch.tensor([oracle.shard_triple(oracle.bf16_to_f64(logits[r, lo:hi]), lo) for r in rows],
                        dtype=torch.float64)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    conf, lse, tok = [], [], []
    for i in range(len(rows)):
        tr = [(float(g[i, 0]), float(g[i, 1]), int(g[i, 2])) for g in gathered]
        c, l, t = oracle.merge_triples(tr)
        conf.append(c), lse.append(l), tok.append(t)
    q.put((rank, np.array(conf), np.array(tok)))
    dist.barrier()
    dist.destroy_process_group()


def test_all_gathered_triples_merge_to_the_unsharded_step():
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted((q.get(timeout=120) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg, inp, rows, logits = _case()
    ref = oracle.step(logits, cfg.V, inp.input_ids, inp.thr, inp.conf_state, cfg.mask_id)
    for rank, conf, tok in results:
        np.testing.assert_array_equal(tok, ref["tok"].reshape(-1)[rows])
        np.testing.assert_allclose(conf, ref["conf"].reshape(-1)[rows], rtol=1e-12)
