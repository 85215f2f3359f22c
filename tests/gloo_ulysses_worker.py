"""Worker for the multi-process check: each rank runs the Ulysses all-to-all the
way the pages describe it -- ``all_to_all_single`` over a process group, heads
scattered and the sequence gathered in rank order (TeleFuser docs
"Communication Architecture", Ulysses section) -- and compares its own
head-group target with the CPU oracle's single-process relayout."""
import os

import torch
import torch.distributed as dist


def ulysses_scatter_heads(x: torch.Tensor, P: int) -> torch.Tensor:
    """[B, Sl, H, D] on this rank -> [B, P*Sl, H/P, D] (this rank's head band)."""
    B, Sl, H, D = x.shape
    Hl = H // P
    send = x.reshape(B, Sl, P, Hl, D).permute(2, 0, 1, 3, 4).contiguous()  # chunk j -> rank j
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv.view(torch.uint8).view(-1), send.view(torch.uint8).view(-1))
    # recv[j] is rank j's tokens of my heads: concatenate in rank order
    return recv.permute(1, 0, 2, 3, 4).reshape(B, P * Sl, Hl, D)


def ulysses_gather_heads(a: torch.Tensor, P: int) -> torch.Tensor:
    """[B, P*Sl, Hl, D] on this rank -> [B, Sl, P*Hl, D] (this rank's tokens, all heads)."""
    B, S, Hl, D = a.shape
    Sl = S // P
    send = a.reshape(B, P, Sl, Hl, D).permute(1, 0, 2, 3, 4).contiguous()  # token block j -> rank j
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv.view(torch.uint8).view(-1), send.view(torch.uint8).view(-1))
    # recv[j] is my tokens of rank j's heads: concatenate along heads in rank order
    return recv.permute(1, 2, 0, 3, 4).reshape(B, Sl, P * Hl, D)


def run(rank, world, port, shapes, result_dir):
    import oracle
    from ulysses_sequence_attention_tf_gb300 import synth

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for i, (B, Sl, H, D, layout, dtype_name) in enumerate(shapes):
            dtype = getattr(torch, dtype_name)
            shards = synth.qkv_shards(world, B, Sl, H, D, dtype, seed=100 + i, layout=layout)
            for key in ("q", "k", "v"):
                mine = ulysses_scatter_heads(shards[key][rank], world)
                want = oracle.scatter(shards[key], world)[rank]
                assert torch.equal(mine.view(torch.uint8), want.view(torch.uint8)), (rank, i, key)
                back = ulysses_gather_heads(mine, world)
                assert torch.equal(back.view(torch.uint8), shards[key][rank].contiguous().view(torch.uint8))
                # oracle gather of the oracle targets agrees with the collective's inverse
                tg = oracle.scatter(shards[key], world)
                assert torch.equal(oracle.gather(tg, world)[rank].view(torch.uint8), back.view(torch.uint8))
        # the chunk exchange: a destination-major payload through all_to_all_single
        for chunk in (16, 48, 4096):
            gen = torch.Generator().manual_seed(7 * chunk)
            payloads = [torch.randint(0, 256, (world, chunk), generator=gen, dtype=torch.uint8) for _ in range(world)]
            recv = torch.empty_like(payloads[rank])
            dist.all_to_all_single(recv.view(-1), payloads[rank].view(-1))
            assert torch.equal(recv, oracle.exchange_chunks(payloads, world)[rank]), (rank, chunk)
        with open(os.path.join(result_dir, f"ok{rank}"), "w") as f:
            f.write("ok")
    finally:
        dist.destroy_process_group()
