"""The EP-group token count ("fix(moe): equalize and align per-rank token
counts for HybridEP dispatch", section "Fix": every rank pads to the aligned
EP-group max), computed by group_num_tokens_per_rank with one all-reduce, on
two gloo ranks on CPU. Each group of counts printed on the page (the
functional test's combos and the DeepSeek-V4-Flash row, five counts per rank)
must give every rank the group max, and its padding the hand-worked value of
tests/golden/padding_vectors.json. Without a process group the local count
comes back unchanged."""
import json
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "padding_vectors.json")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _groups():
    with open(GOLDEN) as f:
        return json.load(f)["group"]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import combine_topk_ids_expert_gb300 as ep
    out = []
    for g in _groups():
        counts = g["counts"]
        share = counts[rank::world]              # the logical ranks this process holds
        local = max(share) if share else 0
        N = ep.group_num_tokens_per_rank(local)
        out.append((N, ep.ep_pad_tokens(N)))
    q.put((rank, out))
    dist.destroy_process_group()


def test_group_max_over_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    for i, g in enumerate(_groups()):
        for rank in (0, 1):
            N, P = res[rank][i]
            assert N == max(g["counts"]), (g["counts"], rank, N)
            assert P == g["padded"], (g["counts"], rank, P, g["cite"])


def test_without_a_process_group_the_local_count():
    import combine_topk_ids_expert_gb300 as ep
    assert not dist.is_initialized()
    assert ep.group_num_tokens_per_rank(13) == 13
    assert ep.ep_pad_tokens(ep.group_num_tokens_per_rank(13)) == 16
