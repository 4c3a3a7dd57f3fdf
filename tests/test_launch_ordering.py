"""Launch ordering against the oracle.  Every kernel of the library is a programmatic
dependent launch, and a decode launch may stream K/V before its grid wait when the host knows
that the cache's previous launch on the stream wrote none of the layer's storage.  These cases
break the patterns that knowledge rests on: two caches interleaved layer by layer on one
stream, ordinary caller kernels between library calls, and one cache's steps alternating
between two streams ordered by events.  Outputs and cache state must match the oracle."""
import numpy as np
import pytest

from harness import Scenario, torch_to_bits

pytestmark = pytest.mark.gpu


def test_two_caches_interleaved_with_caller_kernels():
    import torch
    kw = dict(max_len=512, Hq=8, Hk=2, D=64, W=32, kinds=[1, 0, 1, 0])
    a = Scenario(B=4, seed=101, **kw)
    b = Scenario(B=3, seed=102, **kw)
    junk = torch.ones(1 << 20, device="cuda")
    plan = [([64, 5, 1, 0], [40, 40, 3]), ([1, 1, 1, 1], [1, 1, 1]), ([1, 7, 1, 1], [1, 1, 0]),
            ([1, 1, 1, 1], [1, 1, 1]), ([30, 1, 0, 2], [1, 20, 1]), ([1, 1, 1, 1], [1, 1, 1])]
    for n_a, n_b in plan:
        C = max(max(n_a), max(n_b))
        outs = {id(a): [], id(b): []}
        for layer in range(len(kw["kinds"])):
            for sc, n in ((a, n_a), (b, n_b)):
                outs[id(sc)].append(sc.append_layer(layer, list(range(sc.B)), None, n, C))
                junk.mul_(1.0)          # a caller kernel between library launches
        torch.cuda.synchronize()
        for sc, n in ((a, n_a), (b, n_b)):
            for layer, (q, out) in enumerate(outs[id(sc)]):
                sc.check_outputs(layer, list(range(sc.B)), n, q, torch_to_bits(out))
            sc.cache.advance(list(n))
            sc.lens = [l + k for l, k in zip(sc.lens, n)]
            sc.check_state()


def test_steps_alternating_between_two_streams():
    import torch
    sc = Scenario(B=5, max_len=600, Hq=16, Hk=4, D=128, W=48, kinds=[1, 1, 0, 1], seed=103)
    s0 = torch.cuda.current_stream()
    s1 = torch.cuda.Stream()
    rng = np.random.default_rng(103)
    for step in range(10):
        st = s1 if step % 2 else s0
        st.wait_stream(s0)
        s1.wait_stream(s0)
        with torch.cuda.stream(st):
            if step in (0, 5):
                n = [int(x) for x in rng.integers(1, 65, size=5)]
                sc.step(n, C=64, check_state=True)
            else:
                sc.step([1] * 5, check_state=True)
        s0.wait_stream(st)
