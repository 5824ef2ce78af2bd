"""The masked forms keep each CTA's split-tail items in a shared-memory list
(up to 32) and work out any later item when they reach it.  No workload here
gives a CTA more than a few tail items, so this test builds the same sources
with a list of one item (-DNCP_MAX_CTA_TAIL_ITEMS=1): every tail item after a
CTA's first then takes the worked-out path.  The schedule is the same either
way, so the two builds must give bit-identical outputs."""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs(cuda_lib):
    from non_causal_prefix_gb300 import _build
    variant = ctypes.CDLL(_build.build_variant("taillist1", ["-DNCP_MAX_CTA_TAIL_ITEMS=1"]))
    for name, (res, args) in cuda_lib.SIGNATURES.items():
        fn = getattr(variant, name)
        fn.restype = res
        fn.argtypes = args
    return cuda_lib.load_library(), variant


def ptr(t):
    return t.data_ptr() if t is not None else None


@pytest.mark.parametrize("cid", [6, 9])
def test_tail_list_of_one_matches(libs, cid):
    main, variant = libs
    w = workloads.WORKLOADS[cid]
    ins = [t.cuda() for t in workloads.make_inputs(w)]
    ids = workloads.image_ids(w).cuda()
    valid = workloads.key_valid(w).cuda() if w.kind == "masked_prefix" else None
    outs = []
    for lib in (main, variant):
        out = torch.empty_like(ins[0])
        if w.kind == "block_causal":
            rc = lib.attn_block_causal_fwd(ptr(ins[0]), ptr(ins[1]), ptr(ins[2]), ptr(ids),
                                           ptr(out), w.B, w.Nq, w.H, w.D, None)
        else:
            rc = lib.attn_masked_prefix_fwd(ptr(ins[0]), ptr(ins[1]), ptr(ins[2]), ptr(ins[3]),
                                            ptr(ins[4]), ptr(ids), ptr(valid), w.sm_scale,
                                            ptr(out), w.B, w.Nq, w.Np, w.H, w.D, None)
        assert rc == 0
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.isfinite(outs[0].float()).all()
    assert torch.equal(outs[0], outs[1])
