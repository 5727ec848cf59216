"""The layer split by expert across ranks, on CPU with gloo (world size 2).

The layer shards naturally by expert: the router and the latent projections
are replicated, each rank runs the FFNs of its own expert range on the slots
routed there (the dispatch), and the gate-weighted partial sums meet in one
exchange (the collect) before the up-projection. With the float64 oracle on
every rank and an all-reduce as the exchange, the result must be the
one-rank layer up to summation order: the combine is linear in the expert
outputs, the up-projection linear in c ("The Training and RL Infrastructure
Behind MAI-Thinking-1", section "The model the systems run": the latent is
projected down before dispatch and back up after the combine)."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f64(t):
    return t.float().numpy().astype(np.float64)


def _rank_main(rank, world, port, out_path, cfg_name):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from mixture_experts_layer_router_gb300 import synth
    from oracle import latentmoe_ref as ref

    cfg = synth.CONFIGS[cfg_name]
    w = synth.make_weights(cfg, 4, "cpu")
    x = _f64(synth.make_x(cfg, 4, "cpu"))
    W = ref.OracleWeights.from_stacked(_f64(w["w_r"]), _f64(w["w_dn"]), _f64(w["w_up"]),
                                       _f64(w["w_g"]), _f64(w["w_u"]), _f64(w["w_d"]))
    # replicated: router and latent down-projection
    L = ref.router_logits(x, W.w_r)
    r = ref.route(L, cfg.E, cfg.k)
    z = ref.latent_down(x, W.w_dn)
    # this rank's experts
    per = cfg.E // world
    e0, e1 = rank * per, (rank + 1) * per
    c = np.zeros((cfg.T, cfg.l), dtype=np.float64)
    slots = 0
    for e in range(e0, e1):
        tj = np.argwhere(r["idx"] == e)  # (token, j) pairs routed to e
        if len(tj) == 0:
            continue
        wg, wu, wd = W.expert(e)
        H = ref.swiglu_ffn(z[tj[:, 0]], wg, wu, wd)
        np.add.at(c, tj[:, 0], r["gates"][tj[:, 0], tj[:, 1]][:, None] * H)
        slots += len(tj)
    # the collect: one sum over ranks
    ct = torch.from_numpy(c)
    dist.all_reduce(ct, op=dist.ReduceOp.SUM)
    st = torch.tensor([slots], dtype=torch.int64)
    dist.all_reduce(st, op=dist.ReduceOp.SUM)
    y = ref.latent_up(ct.numpy(), W.w_up)
    full = ref.forward(x, W, cfg.k)["y"]
    err = np.abs(y - full).max() / max(np.abs(full).max(), 1e-300)
    with open(f"{out_path}.{rank}", "w") as f:
        f.write(f"{float(err)!r} {int(st.item())} {cfg.T * cfg.k}")
    dist.barrier()
    dist.destroy_process_group()


def test_expert_split_over_two_ranks_equals_the_layer(tmp_path):
    port = _free_port()
    out = str(tmp_path / "ep")
    mp.start_processes(_rank_main, args=(2, port, out, "tiny"), nprocs=2, start_method="spawn")
    for r in range(2):
        err, slots, want = open(f"{out}.{r}").read().split()
        assert float(err) < 1e-12, err
        assert int(slots) == int(want)  # every slot computed by exactly one rank
