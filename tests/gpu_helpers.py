"""Shared helpers of the GPU parity tests: move workload arrays to the device,
run the library, run the oracle, and compare the two."""

import numpy as np
import torch

import oracle
import speculative_decoding_verification_decode_gb300 as sv

DEV = torch.device("cuda", 0)
MASK_COMPARABLE = ~np.uint32(oracle.NEAR_BOUNDARY | oracle.NEAR_FILTER | oracle.NEAR_DECISION
                             | oracle.DRAW_CERTIFIED | oracle.NEAR_EMPTY
                             | sv.SEQ_EXACT_PATH)


def to_dev(a, dtype=None):
    if a is None:
        return None
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_gpu(wl, mode=None, flags=0, warped=False):
    mode = mode or wl.mode
    cu = to_dev(wl.cu_k)
    k = wl.K if wl.cu_k is not None else None
    if mode == "greedy":
        r = sv.verify_greedy(to_dev(wl.target, wl.dtype), to_dev(wl.tokens), cu, k, flags=flags)
        out = None
    elif mode == "accept":
        r = sv.accept(to_dev(wl.target), to_dev(wl.draft), to_dev(wl.tokens), to_dev(wl.uniforms),
                      cu, k, flags=flags)
        out = None
    else:
        out = None
        if warped:
            out = (torch.full(wl.target.shape, float("nan"), device=DEV),
                   torch.full(wl.draft.shape, float("nan"), device=DEV))
        r = sv.accept_from_logits(to_dev(wl.target, wl.dtype), to_dev(wl.draft, wl.dtype),
                                  to_dev(wl.temperature), to_dev(wl.tokens), to_dev(wl.uniforms),
                                  cu, k, warped_out=out, flags=flags)
    torch.cuda.synchronize()
    res = oracle.Result(r.n_accepted.cpu().numpy(), r.next_token.cpu().numpy(),
                        r.status.cpu().numpy().astype(np.uint32))
    if out is not None:
        return res, (out[0].cpu().numpy(), out[1].cpu().numpy())
    return res


def run_oracle(wl, mode=None):
    mode = mode or wl.mode
    if mode == "greedy":
        return oracle.verify_greedy(wl.target, wl.dtype, wl.tokens, wl.B, wl.K, wl.cu_k)
    if mode == "accept":
        return oracle.accept(wl.target, wl.draft, wl.tokens, wl.uniforms, wl.B, wl.K, wl.cu_k)
    return oracle.accept_from_logits(wl.target, wl.draft, wl.dtype, wl.temperature, wl.tokens,
                                     wl.uniforms, wl.B, wl.K, wl.cu_k)


def compare(gpu, ref, exact_tokens=False):
    """Accepted lengths and statuses must match bit for bit; tokens too,
    except where the oracle flags the draw as near a CDF boundary (1e-5 of
    the total) and does not certify it (a bonus draw from probability rows
    farther than 2^-21 of the total from every step is certified: its id is
    asserted equal whatever the 1e-5 flag says); the ZERO_MASS bit is not
    compared where the oracle flags the residual as near empty.  Returns (number of flagged
    draws, number of flagged draws whose ids differ)."""
    assert np.array_equal(gpu.n_accepted, ref.n_accepted), _first_diff(gpu.n_accepted, ref.n_accepted)
    g_st = gpu.status & MASK_COMPARABLE
    r_st = ref.status & MASK_COMPARABLE
    # a residual within the fp32 band of zero may come out empty or not
    empty = (ref.status & oracle.NEAR_EMPTY) > 0
    g_st = np.where(empty, g_st & ~np.uint32(oracle.ZERO_MASS), g_st)
    r_st = np.where(empty, r_st & ~np.uint32(oracle.ZERO_MASS), r_st)
    assert np.array_equal(g_st, r_st), _first_diff(g_st, r_st)
    near = (ref.status & oracle.NEAR_BOUNDARY) > 0
    same = gpu.next_token == ref.next_token
    certified = (ref.status & oracle.DRAW_CERTIFIED) > 0
    assert (same | ~certified).all(), _first_diff(np.where(certified, gpu.next_token, ref.next_token),
                                                  ref.next_token)
    if exact_tokens:
        assert same.all(), _first_diff(gpu.next_token, ref.next_token)
    else:
        assert (same | near).all(), _first_diff(np.where(near, ref.next_token, gpu.next_token),
                                                ref.next_token)
    return int(near.sum()), int((near & ~same).sum())


def _first_diff(a, b):
    idx = np.flatnonzero(a != b)
    if idx.size == 0:
        return "equal"
    i = idx[0]
    return f"{idx.size} differences; first at sequence {i}: gpu={a[i]} oracle={b[i]}"


def assert_softmax_agreement(gpu, ref, label, mask=None):
    """Accepted lengths against the oracle's own fp64 softmax: equal on every
    sequence the oracle does not flag (NEAR_DECISION: an accept test within
    the fp32 warp's error band of its threshold; NEAR_FILTER: a top-p
    boundary within the filter tolerance).  Prints the agreement and the
    flagged count."""
    sel = np.ones(gpu.n_accepted.shape, bool) if mask is None else np.asarray(mask, bool)
    flagged = (ref.status & np.uint32(oracle.NEAR_DECISION | oracle.NEAR_FILTER)) > 0
    same = gpu.n_accepted == ref.n_accepted
    agree = float(same[sel].mean()) if sel.any() else 1.0
    print(f"{label}: decisions agree with the oracle's fp64 softmax on {agree:.4f} of sequences "
          f"({int((flagged & sel).sum())} flagged near a threshold)")
    bad = sel & ~flagged & ~same
    assert not bad.any(), _first_diff(np.where(bad, gpu.n_accepted, ref.n_accepted), ref.n_accepted)
