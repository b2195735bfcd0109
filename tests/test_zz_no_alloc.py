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
