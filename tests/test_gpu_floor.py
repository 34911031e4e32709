"""pe_latency_floor on the GPU: the empty launch runs, and the dependent
loads end where a walk of the same chain on the host ends (an index
outside the chain continues from entry 0, as the header states)."""
import pytest
import torch

from speculative_decoding_pe_gb300 import _native, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    return _native.load()


def _walk(chain, hops):
    i = 0
    for _ in range(hops):
        i = int(chain[i])
        if not 0 <= i < len(chain):
            i = 0
    return i


@pytest.mark.parametrize("ctas", [1, 608])
def test_latency_floor_follows_the_chain(ctas):
    g = torch.Generator().manual_seed(11)
    n = 1000
    chain = torch.randperm(n, generator=g).to(torch.int32)
    chain[int(chain[0])] = n + 5          # one entry leaves the chain
    dev_chain = chain.cuda()
    out = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    _native.latency_floor(ctas, 0)        # empty launch, nothing written
    _native.latency_floor(ctas, 0, dev_chain, out)
    torch.cuda.synchronize()
    assert int(out.item()) == -7
    for hops in (1, 2, 5, 37, 1000):
        _native.latency_floor(ctas, hops, dev_chain, out)
        torch.cuda.synchronize()
        assert int(out.item()) == _walk(chain.tolist(), hops), hops
