"""spec_verify_sample_noalloc: the sampling entry point that takes no workspace
and allocates nothing (its scratch is a fixed device array in the library).

It must give what spec_verify_sample gives with a caller workspace, call after
call (the fixed scratch is reused, and the part that must start at zero is
cleared by every call), and reject batches whose scratch need exceeds the
array before touching the device.  This file is collected last so that it also
runs after every other GPU test has used the library."""
import ctypes

import numpy as np
import pytest

from speculative_decoding_verification_52_gb300 import binding as B
from speculative_decoding_verification_52_gb300 import build as build_mod
from speculative_decoding_verification_52_gb300 import inputs as gen

NOALLOC_BYTES = 16 << 20


def test_noalloc_rejects_oversized_batch_on_host():
    build_mod.build()
    L = B.lib()
    P = ctypes.c_void_p
    Bn, K, V = 2048, 8, 151936
    assert L.spec_workspace_bytes(Bn, K, V) > NOALLOC_BYTES
    st = L.spec_verify_sample_noalloc(P(1 << 20), B.SPEC_BF16, P(1 << 21), B.SPEC_BF16, B.SPEC_DRAFT_LOGITS,
                                      P(1 << 22), P(1 << 23), 0.7, Bn, K, V, P(1 << 24), P(1 << 25), None)
    assert st == B.SPEC_ERR_UNSUPPORTED
    assert str(NOALLOC_BYTES) in B.last_error()
    # the headline batch fits
    assert L.spec_workspace_bytes(256, 5, 128256) <= NOALLOC_BYTES


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", ["headline", "zipf"])
def test_noalloc_matches_workspace_entry_point_twice(orc, cfg):
    import torch

    import speculative_decoding_verification_52_gb300 as sv
    from gpu_util import DEV, compare_sample, dev_tensor, f32, i32, oracle_sample

    if cfg == "headline":
        batch = gen.config_headline(seqs=list(range(64)))
    else:
        batch = gen.config_zipf(T=1.0, B=32)
    Bn, K = batch.B, batch.K
    target = dev_tensor(batch.target, batch.dtype)
    draft = dev_tensor(batch.draft, batch.draft_dtype)
    tok, uni = i32(batch.draft_tokens), f32(batch.uniforms)

    ref_out, ref_n = sv.spec_verify_sample(target, draft, tok, uni, batch.T)
    ref_out, ref_n = ref_out.cpu().numpy(), ref_n.cpu().numpy()

    out = torch.full((Bn, K + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((Bn,), -7, dtype=torch.int32, device=DEV)
    for call in range(2):
        sv.spec_verify_sample_noalloc(target, draft, tok, uni, batch.T, out_tokens=out, num_accepted=nacc)
        torch.cuda.synchronize()
        o, n = out.cpu().numpy(), nacc.cpu().numpy()
        # same kernel, same inputs: the decisions agree exactly with the workspace entry point
        np.testing.assert_array_equal(n, ref_n, err_msg=f"call {call}: num_accepted differs")
        np.testing.assert_array_equal(o, ref_out, err_msg=f"call {call}: out_tokens differ")
        # and both follow the oracle under the sampling-mode comparison rule
        compare_sample(o, n, oracle_sample(orc, batch))
        out.fill_(-7)
        nacc.fill_(-7)


@pytest.mark.gpu
def test_noalloc_greedy_twice_matches_greedy_entry_point(orc):
    """T = 0 sends the fixed scratch through the greedy chain kernel, whose
    layout differs from the sampling kernel's: two calls in a row must match
    spec_verify_greedy and the oracle bit for bit."""
    import torch

    import speculative_decoding_verification_52_gb300 as sv
    from gpu_util import DEV, dev_tensor, i32

    batch = gen.config_greedy(seqs=list(range(96)))
    Bn, K = batch.B, batch.K
    target = dev_tensor(batch.target, batch.dtype)
    tok = i32(batch.draft_tokens)
    ro, rn = orc.verify_greedy(batch.target, batch.dtype, batch.draft_tokens)
    go, gn = sv.spec_verify_greedy(target, tok)
    np.testing.assert_array_equal(gn.cpu().numpy(), rn)
    np.testing.assert_array_equal(go.cpu().numpy(), ro)
    # the sampling signature at T = 0: draft and uniforms are not read
    out = torch.full((Bn, K + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((Bn,), -7, dtype=torch.int32, device=DEV)
    for call in range(2):
        sv.spec_verify_sample_noalloc(target, None, tok, None, 0.0, out_tokens=out, num_accepted=nacc)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(nacc.cpu().numpy(), rn, err_msg=f"call {call}: num_accepted differs")
        np.testing.assert_array_equal(out.cpu().numpy(), ro, err_msg=f"call {call}: out_tokens differ")
        out.fill_(-7)
        nacc.fill_(-7)


@pytest.mark.gpu
def test_noalloc_sampling_then_greedy_then_sampling(orc):
    """Calls of the two kernels share the fixed scratch in turn: what one
    leaves in it (control words, counters, queue slots) must not leak into
    the next call of the other."""
    import torch

    import speculative_decoding_verification_52_gb300 as sv
    from gpu_util import DEV, compare_sample, dev_tensor, f32, i32, oracle_sample

    sb = gen.config_headline(seqs=list(range(48)))
    gb = gen.config_greedy(seqs=list(range(48)))
    st, sd = dev_tensor(sb.target, sb.dtype), dev_tensor(sb.draft, sb.draft_dtype)
    stok, suni = i32(sb.draft_tokens), f32(sb.uniforms)
    gt, gtok = dev_tensor(gb.target, gb.dtype), i32(gb.draft_tokens)
    sref = oracle_sample(orc, sb)
    ro, rn = orc.verify_greedy(gb.target, gb.dtype, gb.draft_tokens)
    out = torch.empty((sb.B, sb.K + 1), dtype=torch.int32, device=DEV)
    nacc = torch.empty((sb.B,), dtype=torch.int32, device=DEV)
    for step in ("sample", "greedy", "sample", "greedy"):
        out.fill_(-7)
        nacc.fill_(-7)
        if step == "sample":
            sv.spec_verify_sample_noalloc(st, sd, stok, suni, sb.T, out_tokens=out, num_accepted=nacc)
            torch.cuda.synchronize()
            compare_sample(out.cpu().numpy(), nacc.cpu().numpy(), sref)
        else:
            sv.spec_verify_sample_noalloc(gt, None, gtok, None, 0.0, out_tokens=out, num_accepted=nacc)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(nacc.cpu().numpy(), rn)
            np.testing.assert_array_equal(out.cpu().numpy(), ro)
