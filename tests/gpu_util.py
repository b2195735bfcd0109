"""Helpers for the GPU parity tests: numpy batches -> device tensors, CUDA
calls through the binding, and the comparison rule against the oracle."""
import numpy as np
import torch

import speculative_decoding_verification_52_gb300 as sv

DEV = torch.device("cuda:0")


def dev_tensor(x: np.ndarray, dtype: str) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if dtype == "bf16":
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(x.astype(np.float32, copy=False)).to(DEV)


def i32(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(DEV)


def f32(x) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)


def gpu_sample(batch, T=None, draft_dtype=None):
    T = batch.T if T is None else T
    ddt = batch.draft_dtype if draft_dtype is None else draft_dtype
    draft = dev_tensor(batch.draft, ddt) if batch.K > 0 else None
    out, n = sv.spec_verify_sample(dev_tensor(batch.target, batch.dtype), draft,
                                   i32(batch.draft_tokens) if batch.K > 0 else None,
                                   f32(batch.uniforms), T,
                                   draft_kind="probs" if batch.draft_is_probs else "logits")
    return out.cpu().numpy(), n.cpu().numpy()


def oracle_sample(orc, batch, T=None):
    T = batch.T if T is None else T
    return orc.verify_sample(batch.target, batch.dtype, batch.draft, batch.draft_dtype, batch.draft_is_probs,
                             batch.draft_tokens, batch.uniforms, T)


def compare_sample(out, n, ref, stats=None):
    """Bit-exact comparison except after decisions the oracle flags as within
    1e-6 of flipping: a near accept test at t excludes slots >= t and the
    accept count; a near CDF boundary excludes only the drawn token.
    Returns the number of flagged sequences; asserts on any other mismatch.
    `stats` (a dict) receives flagged / flagged_mismatch counts."""
    na, nc = ref["near_accept"], ref["near_cdf"]
    ro, rn = ref["out_tokens"], ref["num_accepted"]
    flagged = flagged_mismatch = 0
    bad = []
    for b in range(len(rn)):
        if na[b] >= 0:
            flagged += 1
            t = na[b]
            if not (out[b, :t] == ro[b, :t]).all():
                bad.append(b)
            if n[b] != rn[b] or not (out[b] == ro[b]).all():
                flagged_mismatch += 1
            continue
        if nc[b]:
            flagged += 1
            m = rn[b]
            if n[b] != m or not (out[b, :m] == ro[b, :m]).all() or not (out[b, m + 1:] == ro[b, m + 1:]).all():
                bad.append(b)
            if out[b, m] != ro[b, m]:
                flagged_mismatch += 1
            continue
        if n[b] != rn[b] or not (out[b] == ro[b]).all():
            bad.append(b)
    assert not bad, f"{len(bad)} sequences differ from the oracle, first {bad[:5]}: " \
                    f"gpu n={n[bad[0]]} {out[bad[0]].tolist()} oracle n={rn[bad[0]]} {ro[bad[0]].tolist()}"
    if stats is not None:
        stats.update(flagged=flagged, flagged_mismatch=flagged_mismatch, total=len(rn))
    return flagged
