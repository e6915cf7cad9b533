"""Cache views with a different physical layout.

The C ABI takes element strides, so a cache whose memory is token-major
([R, T, L, H, d]: all heads of a token adjacent, as paged serving caches keep
them) is passed as a strided [R, L, H, T, d] view.  The whole chain must give
bit-identical results to the default head-major layout: the kernels read the
same values in the same order, only the addresses differ.
"""
import dataclasses

import pytest
import torch

from agent_shared_context_gb300 import synth

pytestmark = pytest.mark.gpu


def _token_major(x):
    """Same logical [R, L, H, T, d] tensor stored as [R, T, L, H, d]."""
    return x.permute(0, 3, 1, 2, 4).contiguous().permute(0, 2, 3, 1, 4)


@pytest.mark.parametrize("name", ["bf16", "f32"])
def test_token_major_layout_is_bit_identical(name):
    from agent_shared_context_gb300.chain import ChainRunner
    if name == "bf16":
        wl = synth.scaled(synth.workload("concurrent"), L=2, H=2, R=2, seg_len=[256, 205], pf=16,
                          fallback_frac=0.25)
    else:
        wl = synth.scaled(synth.workload("tiny"), L=1, H=2, R=1, seg_len=[200, 56], pf=8,
                          n_agents=3, build_slot=-1)
    inp = synth.generate(wl, device="cuda")
    alt = dataclasses.replace(inp, exact_K=[_token_major(t) for t in inp.exact_K],
                              exact_V=[_token_major(t) for t in inp.exact_V])
    assert alt.exact_K[0].stride(3) == wl.L * wl.H * wl.d          # token stride
    assert torch.equal(alt.exact_K[1], inp.exact_K[1])
    a = ChainRunner(wl, inp, device="cuda")
    b = ChainRunner(wl, alt, device="cuda")
    assert b.edges[1].out_K.stride() == alt.exact_K[1].stride()     # outputs keep the layout
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert int(a.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    for j in range(1, wl.edges + 1):
        ea, eb = a.edges[j], b.edges[j]
        for key in ("out_K", "out_V", "weights", "best", "score", "fallback"):
            assert torch.equal(getattr(ea, key), getattr(eb, key)), (j, key)
