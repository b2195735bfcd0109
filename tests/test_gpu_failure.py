"""Bounded waits on the GPU: a wait that nothing satisfies runs out, the call
reports -2 for every sequence, and the context stays usable (a normal call
right after it matches the oracle).  No fault, trap or hang is involved: the
test hook makes one sequence's accept scan wait for a sweep unit that is
never produced, with every device-side wait limited to 2 ms."""
import time

import numpy as np
import pytest
import torch

import gpu_util as gu
import speculative_decoding_verification_52_gb300 as sv
from speculative_decoding_verification_52_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_minus_two_and_context_survives(orc):
    b = gen.config_headline(B=16, V=4096)
    t, d = gu.dev_tensor(b.target, "bf16"), gu.dev_tensor(b.draft, "bf16")
    tok, uni = gu.i32(b.draft_tokens), gu.f32(b.uniforms)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    out, n = sv.spec_debug_stall(t, d, tok, uni, b.T, stall_b=5, timeout_us=2000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert (n.cpu().numpy() == -2).all()
    assert (out.cpu().numpy() == -1).all()
    assert dt < 5.0, f"the bounded waits took {dt:.2f} s"
    # the same context and a fresh call: normal results
    out2, n2 = sv.spec_verify_sample(t, d, tok, uni, b.T)
    ref = orc.verify_sample(b.target, "bf16", b.draft, "bf16", False, b.draft_tokens, b.uniforms, b.T)
    gu.compare_sample(out2.cpu().numpy(), n2.cpu().numpy(), ref)


def test_stall_hook_rejects_bad_arguments():
    b = gen.config_headline(B=4, V=1024)
    t, d = gu.dev_tensor(b.target, "bf16"), gu.dev_tensor(b.draft, "bf16")
    tok, uni = gu.i32(b.draft_tokens), gu.f32(b.uniforms)
    with pytest.raises(sv.SpecError):
        sv.spec_debug_stall(t, d, tok, uni, b.T, stall_b=4, timeout_us=2000)
    with pytest.raises(sv.SpecError):
        sv.spec_debug_stall(t, d, tok, uni, b.T, stall_b=0, timeout_us=10)
