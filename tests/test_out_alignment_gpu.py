"""Output rows at any address the caller chooses.

The merge writes each lane's share of an output row with one vector store
when the caller's `out` pointer is aligned for it, and element by element
otherwise (the boundary asks no alignment of `out`).  The same call into an
aligned buffer and into one shifted by a single element runs the same plan
and the same arithmetic, so the two outputs must agree bit for bit; the
element in front of the shifted buffer must stay untouched.  Cases: the
tensor-core kernel (bf16, head_dim 128: 8-byte stores) and the SIMT kernel
(fp32 and bf16 with head_dim 64: 8- and 4-byte stores), on ragged blocks.
"""
import pytest
import torch

from concurrent_shared_kv_gb300 import workloads as wl
from tests import harness as H

pytestmark = pytest.mark.gpu


def _ragged_bf16(head_dim: int) -> wl.Workload:
    return wl.Workload(f"bf16 W3 Hq8/Hkv2 D{head_dim} common700 blocks130/1/64", "bf16", 1, 3, 8, 2,
                       head_dim, 1e4, 1, [700], [[130, 1, 64]], seed=1201)


CASES = {
    "tc-bf16-d128": lambda: _ragged_bf16(128),
    "simt-bf16-d64": lambda: _ragged_bf16(64),
    "simt-f32-d64": wl.tiny_f32,
}


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("name", list(CASES))
def test_shifted_output_matches_aligned_bit_for_bit(name):
    w = CASES[name]()
    c = H.host_case(w) if w.dtype == "f32" else H.device_case(w, 0)
    s = c.session()
    ref_out, ref_lse = s.decode(c.q, c.k, c.v)
    torch.cuda.synchronize()
    assert torch.isfinite(ref_out).all()

    buf = torch.full((ref_out.numel() + 1,), float("nan"), dtype=ref_out.dtype, device=ref_out.device)
    out = buf[1:].view(ref_out.shape)
    # not aligned for two elements, so no vector store of any width applies
    assert out.data_ptr() % (2 * out.element_size()) != 0
    lse = torch.full_like(ref_lse, float("nan"))
    s.decode(c.q, c.k, c.v, out=out, lse=lse)
    torch.cuda.synchronize()

    assert torch.equal(_bits(out), _bits(ref_out))
    assert torch.equal(lse, ref_lse)
    assert torch.isnan(buf[0]).item()
