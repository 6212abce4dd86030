"""Chunk appends whose work is spread unevenly over a call: sequences that take
nothing, one token, a few tokens past a page boundary, or hundreds of tokens,
from lengths that are not multiples of the key group, so that the value tokens
leaving the window per (sequence, kv head) range from none to more than a
staged batch of them. The append kernel lays its items on a work line (a ring
item weighed by its leaving tokens) and cuts it into one slice per CTA; the
pages and rings of every sequence must still equal the oracle's image bit for
bit, for both code widths."""
import dataclasses

import numpy as np
import pytest

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario

pytestmark = pytest.mark.gpu

SIZES = (0, 0, 1, 1, 2, 5, 17, 31, 33, 64, 100, 129, 300, 700)


@pytest.mark.parametrize("bits", [4, 2])
def test_skewed_ragged_appends_match_the_oracle(bits):
    w = dataclasses.replace(inp.WORKLOADS["qwen2.5-1.5b"], residual_v=128)
    rng = np.random.default_rng(40 + bits)
    B, steps = 24, 4
    lens = [int(x) for x in rng.integers(0, 600, B)]
    plan = [[int(rng.choice(SIZES)) for _ in range(B)] for _ in range(steps)]
    extra = max(sum(p[b] for p in plan) for b in range(B))
    sc = Scenario(w, 40 + bits, lens, extra_tokens=extra, bits=bits)
    sc.fill()
    for step, news in enumerate(plan):
        sc.cur = sc.append(0, news, 1 + step)
        rc, detail = sc.cache.status()
        assert rc == 0, (s4.s4kv_strerror(rc), detail)
    for b in range(B):
        sc.check_bytes(0, b)
