"""The compressed tier's host encoder (in the library, no GPU needed) against the oracle codec.

The library's stream must equal the oracle's encoding byte for byte, and the oracle must decode it to the
input: over block boundaries, odd lengths, quantised-weight-like and uniform nibbles, and constant bytes.
"""
import pytest

import oracle.ans as A
from int4_grouped_expert_router_gb300 import synth


@pytest.fixture(scope="module")
def B():
    from int4_grouped_expert_router_gb300.build import build
    build()
    from int4_grouped_expert_router_gb300 import binding
    return binding


CASES = [(1, "gauss"), (77, "gauss"), (4096, "gauss"), (12289, "gauss"), (6000, "uniform"), (5000, "const")]


@pytest.mark.parametrize("n,kind", CASES, ids=[f"{k}-{n}" for n, k in CASES])
def test_library_encoder_equals_oracle(B, n, kind):
    if kind == "gauss":
        data = bytes(synth.gaussian_nibble_bytes(synth.stream_seed(97, n), n, 2.5))
    elif kind == "uniform":
        data = bytes(synth.random_bytes(synth.stream_seed(98, n), n))
    else:
        data = bytes([0x79]) * n
    got = B.coli_ans_encode_host(data)
    assert got == A.encode(data)
    assert A.decode(got) == data
    if kind == "gauss" and n >= 4096:
        assert len(got) < 0.95 * n  # quantised-weight-like nibbles compress (entropy about 3.4 bits a nibble)
    if kind == "uniform":
        assert len(got) > n  # uniform nibbles do not
