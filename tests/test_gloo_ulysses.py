"""Multi-process pin of the relayout: P gloo ranks on the CPU run the pages'
all_to_all_single formulation of the Ulysses exchange; every rank's head-group
target must equal the oracle's bit for bit, and the inverse exchange must
restore the shard."""
import socket

import pytest
import torch.multiprocessing as mp

import gloo_ulysses_worker

SHAPES = [
    (1, 6, 8, 16, "contiguous", "bfloat16"),
    (2, 5, 8, 8, "fused", "float16"),
    (1, 3, 16, 4, "v_strided", "float32"),
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_all_to_all_matches_oracle(world, tmp_path):
    mp.spawn(gloo_ulysses_worker.run, args=(world, _free_port(), SHAPES, str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        assert (tmp_path / f"ok{r}").exists()
