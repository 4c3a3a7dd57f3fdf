"""A mixed scenario whose outputs and cache state are written to an .npz file; run by
tests/test_pdl_equivalence.py in a child process under different launch settings."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
from harness import Scenario, torch_to_bits  # noqa: E402


def run(path):
    import torch
    kinds = [1, 0, 1, 1, 0]                       # sliding and global layers, back to back
    sc = Scenario(B=12, max_len=2048, Hq=16, Hk=4, D=128, W=96, kinds=kinds, seed=91)
    outs = []
    rng = np.random.default_rng(91)
    sc.step([64] * 12, C=64, check=False)
    for step in range(12):
        if step % 4 == 3:                          # chunk rows, idle rows, resets
            n = [int(x) for x in rng.integers(0, 40, size=12)]
            res = sc.step(n, C=40, resets=[int(rng.integers(0, 12))], check=False)
        else:                                      # decode steps: sliding -> sliding launches
            res = sc.step([1] * 12, check=False)
        outs += [torch_to_bits(o) for _, o in res]
    sc.copy_rows(sc, src_rows=[0], dst_rows=[5])  # a copy, then decodes after it
    for _ in range(3):
        outs += [torch_to_bits(o) for _, o in sc.step([1] * 12, check=False)]
    torch.cuda.synchronize()
    # the live state only: positions below lens of a global layer, ring slots holding a
    # live position (pads all land on one scratch slot per row, in scheduling order)
    state = []
    for layer, kind in enumerate(kinds):
        for x in sc.cache.storage(layer):
            bits = torch_to_bits(x)
            for b, L in enumerate(sc.cache.lens):
                if kind == 0:
                    slots = np.arange(L)
                else:
                    ring = oracle.ring_positions(L, sc.cache.R)
                    slots = np.nonzero(ring >= 0)[0]
                state.append(bits[b][:, slots])
    np.savez(path, *outs, *state, lens=np.array(sc.cache.lens))


if __name__ == "__main__":
    run(sys.argv[1])
