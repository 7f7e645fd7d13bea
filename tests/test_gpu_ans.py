"""The compressed tier's decoder on the GPU: bit-exact against the input and the oracle codec.

Streams of quantised-weight-like nibbles (one block, several blocks, a short last block, a 6 MB expert
tensor), uniform nibbles and constant bytes are uploaded, decoded by one warp per block, and compared byte
for byte with the input; the stored sizes equal the host encoder's.
"""
import numpy as np
import pytest
import torch

import oracle.ans as A
from int4_grouped_expert_router_gb300 import binding as B
from int4_grouped_expert_router_gb300 import synth
from gpu_util import Ctx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = Ctx()
    yield c.ctx
    c.close()


CASES = [(1, "gauss"), (4096, "gauss"), (4097, "gauss"), (100003, "gauss"), (2048 * 3072, "gauss"),
         (70000, "uniform"), (9000, "const")]


@pytest.mark.parametrize("n,kind", CASES, ids=[f"{k}-{n}" for n, k in CASES])
def test_decode_is_exact(ctx, n, kind):
    if kind == "gauss":
        data = synth.gaussian_nibble_bytes(synth.stream_seed(99, n), n, 2.5)
    elif kind == "uniform":
        data = synth.random_bytes(synth.stream_seed(98, n), n)
    else:
        data = np.full(n, 0x86, np.uint8)
    h = B.coli_ans_upload(ctx, data.tobytes())
    try:
        raw, stored = B.coli_ans_info(ctx, h)
        assert raw == n
        if n <= 100003:
            assert stored == len(A.encode(data.tobytes()))
        out = torch.full((n,), 0x5A, dtype=torch.uint8, device="cuda")
        B.coli_ans_decode(ctx, h, out)
        assert B.coli_check_error(ctx) == 0, B.coli_last_error(ctx)
        assert np.array_equal(out.cpu().numpy(), data)
        print(kind, n, "stored/raw", round(stored / n, 4))
    finally:
        B.coli_ans_free(ctx, h)
