"""GPU parity: the CUDA path against the FP64 oracle on the same seeded bf16
inputs, through the C ABI (via the ctypes binding).

Small shapes span several 128-row tiles and ragged tails in every length
(N, Nq, Np, Nc); the five synthetic workloads run at full size, compared in
full where the oracle finishes in seconds and on sampled rows otherwise.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_parity, bf16_round, sample_rows, stats

pytestmark = pytest.mark.gpu


def to_dev(ts):
    return [t.cuda() for t in ts]


def bits(ts):
    return [workloads.bf16_bits(t) for t in ts]


def gpu_dense(ncp, q, k, v):
    out = torch.empty_like(q)
    ncp.attn_dense_fwd(q, k, v, out)
    torch.cuda.synchronize()
    return out


def gpu_prefix(ncp, q, kp, vp, kc, vc):
    out = torch.empty_like(q)
    ncp.attn_prefix_fwd(q, kp, vp, kc, vc, out)
    torch.cuda.synchronize()
    return out


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


SMALL_DENSE = [  # (B, N, H, D)
    (1, 1, 1, 64), (1, 2, 1, 128), (1, 127, 2, 64), (1, 128, 2, 128), (1, 129, 2, 64),
    (2, 255, 3, 128), (1, 256, 1, 64), (1, 257, 2, 128), (2, 300, 2, 64), (1, 513, 3, 128),
    (1, 1000, 2, 128), (1, 1000, 2, 64),
]


@pytest.mark.parametrize("B,N,H,D", SMALL_DENSE)
def test_dense_small(cuda_lib, oracle_mod, B, N, H, D):
    w = workloads.custom("dense", B, N, N, H, D)
    ins = workloads.make_inputs(w, seed_base=7000 + N + D)
    out = gpu_dense(cuda_lib, *to_dev(ins))
    ref = oracle_mod.dense_attention(*bits(ins))
    assert_parity(f64(out), ref, w.describe())


SMALL_PREFIX = [  # (B, Nq, Np, Nc, H, D)
    (1, 128, 0, 128, 2, 128), (1, 128, 1, 128, 2, 128), (1, 129, 127, 129, 2, 128),
    (2, 200, 128, 200, 2, 128), (1, 300, 129, 300, 1, 128), (1, 64, 1024, 64, 2, 128),
    (1, 257, 300, 100, 2, 64), (1, 100, 5, 700, 2, 64), (2, 1, 1, 1, 3, 128),
    (1, 384, 256, 384, 2, 128),
]


@pytest.mark.parametrize("B,Nq,Np,Nc,H,D", SMALL_PREFIX)
def test_prefix_small(cuda_lib, oracle_mod, B, Nq, Np, Nc, H, D):
    g = workloads.custom("prefix", B, Nq, Nc, H, D, Np=Np)
    q = workloads.randn_bf16((B, Nq, H, D), 1.0, 9100 + Np)
    kp = workloads.randn_bf16((B, Np, H, D), 1.0, 9200 + Np)
    vp = workloads.randn_bf16((B, Np, H, D), 1.0, 9300 + Np)
    kc = workloads.randn_bf16((B, Nc, H, D), 1.0, 9400 + Nc)
    vc = workloads.randn_bf16((B, Nc, H, D), 1.0, 9500 + Nc)
    dq, dkp, dvp, dkc, dvc = to_dev([q, kp, vp, kc, vc])
    if Np == 0:
        dkp = dvp = None
    out = gpu_prefix(cuda_lib, dq, dkp, dvp, dkc, dvc)
    ref = oracle_mod.prefix_attention(*bits([q]), *(bits([kp, vp]) if Np else (None, None)),
                                      *bits([kc, vc]))
    assert_parity(f64(out), ref, g.describe())


# Shapes with fewer work units than SMs and many key tiles: the last (here the
# only) round of units is cut into key-range pieces merged through the
# workspace.  The prefix case cuts across the prefix/current boundary.
SPLIT_CASES = [  # (kind, B, Nq, Np, Nc, H, D)
    ("dense", 1, 2048, 0, 2048, 3, 128), ("dense", 1, 4096, 0, 4096, 1, 64),
    ("dense", 2, 1000, 0, 1000, 1, 128), ("prefix", 1, 512, 640, 512, 2, 128),
    ("prefix", 1, 200, 1100, 300, 2, 64),
]


def split_inputs(kind, B, Nq, Np, Nc, H, D, seed):
    shapes = [(B, Nq, H, D)]
    if kind == "prefix":
        shapes += [(B, Np, H, D)] * 2
    shapes += [(B, Nc, H, D)] * 2
    return [workloads.randn_bf16(s, 1.0, seed + i) for i, s in enumerate(shapes)]


def run_split(ncp, kind, dev):
    if kind == "dense":
        return gpu_dense(ncp, *dev)
    return gpu_prefix(ncp, *dev)


@pytest.mark.parametrize("case", SPLIT_CASES)
def test_split_units(cuda_lib, oracle_mod, case):
    kind, B, Nq, Np, Nc, H, D = case
    ins = split_inputs(kind, B, Nq, Np, Nc, H, D, 9900 + Nq + Np)
    out = run_split(cuda_lib, kind, to_dev(ins))
    if kind == "dense":
        ref = oracle_mod.dense_attention(*bits(ins))
    else:
        ref = oracle_mod.prefix_attention(*bits(ins))
    assert_parity(f64(out), ref, str(case))


def test_split_units_deterministic_and_per_stream(cuda_lib):
    """The merge sums the pieces in a fixed order: repeated calls are
    bit-identical; calls on two streams at once use separate workspaces."""
    kind, B, Nq, Np, Nc, H, D = SPLIT_CASES[0]
    ins = to_dev(split_inputs(kind, B, Nq, Np, Nc, H, D, 9950))
    first = run_split(cuda_lib, kind, ins)
    for _ in range(3):
        assert torch.equal(run_split(cuda_lib, kind, ins), first)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(ins[0]) for _ in streams]
    torch.cuda.synchronize()
    for _ in range(4):
        for s, o in zip(streams, outs):
            cuda_lib.attn_dense_fwd(*ins, o, stream=s)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, first)


def test_prefix_equals_concat_bitwise(cuda_lib):
    """With Np a multiple of the 128-key tile, walking the two segments visits
    the same tiles in the same order as one concatenated key set, so the
    outputs are bit-identical (definition: keys = cat(K_prefix, K_current))."""
    B, Nq, Np, Nc, H, D = 1, 300, 256, 300, 2, 128
    ts = [workloads.randn_bf16(s, 1.0, 9600 + i) for i, s in enumerate(
        [(B, Nq, H, D), (B, Np, H, D), (B, Np, H, D), (B, Nc, H, D), (B, Nc, H, D)])]
    q, kp, vp, kc, vc = to_dev(ts)
    a = gpu_prefix(cuda_lib, q, kp, vp, kc, vc)
    b = gpu_prefix(cuda_lib, q, None, None, torch.cat([kp, kc], 1).contiguous(),
                   torch.cat([vp, vc], 1).contiguous())
    assert torch.equal(a, b)


def test_deterministic_and_inputs_unchanged(cuda_lib):
    w = workloads.custom("dense", 2, 700, 700, 4, 128)
    ins = to_dev(workloads.make_inputs(w, seed_base=9700))
    before = [t.clone() for t in ins]
    a = gpu_dense(cuda_lib, *ins)
    b = gpu_dense(cuda_lib, *ins)
    assert torch.equal(a, b)
    for x, y in zip(ins, before):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_side_stream(cuda_lib, oracle_mod):
    w = workloads.custom("dense", 1, 300, 300, 2, 64)
    ins = workloads.make_inputs(w, seed_base=9800)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q, k, v = to_dev(ins)
        out = torch.empty_like(q)
        cuda_lib.attn_dense_fwd(q, k, v, out, stream=s)
    s.synchronize()
    assert_parity(f64(out), oracle_mod.dense_attention(*bits(ins)), "side stream")


@pytest.mark.parametrize("D", [128, 64])
def test_bounded_wait_reports_timeout(cuda_lib, oracle_mod, D):
    """A wait that can never complete (the loader skips one value tile on
    purpose) ends with ATTN_ERR_TIMEOUT instead of a hang, and the context
    stays usable for the next call.  D = 128 loads K and V into ring slots of
    their own; D = 64 loads them into one entry, whose full barrier then never
    completes."""
    w = workloads.custom("dense", 1, 256, 256, 1, D)
    ins = workloads.make_inputs(w, seed_base=9900)
    q, k, v = to_dev(ins)
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    cuda_lib.debug_set_fault(1, 50_000)
    try:
        out = torch.empty_like(q)
        cuda_lib.attn_dense_fwd(q, k, v, out)
        rc, info = cuda_lib.device_status()
    finally:
        cuda_lib.debug_set_fault(0, 0)
    assert rc == cuda_lib.ATTN_ERR_TIMEOUT
    assert info & 0xff != 0
    out = gpu_dense(cuda_lib, q, k, v)
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    assert_parity(f64(out), oracle_mod.dense_attention(*bits(ins)), "after timeout")


def test_timeout_in_split_launch_leaves_next_call_exact(cuda_lib, oracle_mod):
    """A launch with a split tail that gives up part-way: block 0 times out in
    its first unit and never reaches its tail pieces, so the other pieces of
    those tail units stay counted in.  The next launch on the same workspace
    tags its counters with a new epoch and must give the same bits as before
    the fault."""
    w = workloads.WORKLOADS[2]   # 3 whole rounds, then 56 units split over the SMs
    ins = workloads.make_inputs(w)
    q, k, v = to_dev(ins)
    good = gpu_dense(cuda_lib, q, k, v)
    assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
    cuda_lib.debug_set_fault(1, 50_000)
    try:
        cuda_lib.attn_dense_fwd(q, k, v, torch.empty_like(q))
        rc, _ = cuda_lib.device_status()
    finally:
        cuda_lib.debug_set_fault(0, 0)
    assert rc == cuda_lib.ATTN_ERR_TIMEOUT
    for _ in range(2):
        out = gpu_dense(cuda_lib, q, k, v)
        assert cuda_lib.device_status()[0] == cuda_lib.ATTN_OK
        assert torch.equal(out, good)
    rows = sample_rows(w.B, w.Nq, w.H, n_random=200, seed=22)
    ref = oracle_mod.dense_attention_rows(*bits(ins), rows)
    assert_parity(f64(out).reshape(-1, w.D)[rows], ref, "after a split-launch timeout")


@pytest.mark.parametrize("B,N,H,D", [(1, 1000, 2, 128), (2, 300, 3, 64), (1, 4096, 32, 128)])
def test_output_aligned_16_not_32(cuda_lib, oracle_mod, B, N, H, D):
    """An output 16 bytes past a 32-byte boundary (the entry points ask for 16)
    takes the 16-byte stores: bit-identical to an aligned output, and exact
    against the oracle.  The last shape splits units across SMs, so the
    merge's writes are covered too."""
    w = workloads.custom("dense", B, N, N, H, D)
    ins = workloads.make_inputs(w, seed_base=7600 + N + D)
    q, k, v = to_dev(ins)
    ref_out = gpu_dense(cuda_lib, q, k, v)
    assert ref_out.data_ptr() % 32 == 0
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(q.shape)
    assert out.data_ptr() % 32 == 16
    cuda_lib.attn_dense_fwd(q, k, v, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)
    if N * H <= 2000:
        assert_parity(f64(out), oracle_mod.dense_attention(*bits(ins)), w.describe())
    else:
        rows = sample_rows(B, N, H, 60, seed=7601)
        ref = oracle_mod.dense_attention_rows(*bits(ins), rows)
        assert_parity(f64(out).reshape(-1, D)[rows], ref, w.describe())


def test_binding_rejects_bad_tensors(cuda_lib):
    q = torch.zeros(1, 128, 2, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        cuda_lib.attn_dense_fwd(q.float(), q, q, torch.empty_like(q))
    with pytest.raises(ValueError):
        cuda_lib.attn_dense_fwd(q, q[:, :64], q, torch.empty_like(q))
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.attn_dense_fwd(q, q, q, q)      # out aliases the inputs
    assert e.value.status == cuda_lib.ATTN_ERR_ALIAS


# --------------------------------------------------------------------------
# The five synthetic workloads at full size, in the bench's launch
# configuration (one call of the C ABI over the whole batch).
# --------------------------------------------------------------------------

def run_workload(ncp, w, ins_dev):
    if w.kind == "dense":
        return gpu_dense(ncp, *ins_dev)
    return gpu_prefix(ncp, *ins_dev)


@pytest.mark.parametrize("cid", [1, 2, 4])
def test_workload_full(cuda_lib, oracle_mod, cid):
    w = workloads.WORKLOADS[cid]
    ins = workloads.make_inputs(w)
    out = run_workload(cuda_lib, w, to_dev(ins))
    if w.kind == "dense":
        ref = oracle_mod.dense_attention(*bits(ins))
    else:
        ref = oracle_mod.prefix_attention(*bits(ins))
    s = assert_parity(f64(out), ref, w.describe())
    # The rounded oracle is reported for context: bf16 output rounding alone.
    s_r = stats(bf16_round(ref), ref)
    print(w.name, s, "bf16(oracle):", s_r)


@pytest.mark.parametrize("cid", [3, 5])
def test_workload_sampled(cuda_lib, oracle_mod, cid):
    w = workloads.WORKLOADS[cid]
    ins = workloads.make_inputs(w)
    out = run_workload(cuda_lib, w, to_dev(ins))
    rows = sample_rows(w.B, w.Nq, w.H, n_random=400, seed=cid)
    got = f64(out).reshape(-1, w.D)[rows]
    ref = oracle_mod.dense_attention_rows(*bits(ins), rows)
    s = assert_parity(got, ref, w.describe())
    print(w.name, s)
    if cid == 5:
        # Negative controls on the same rows: an all-zero output and the mean
        # of V (a kernel blind to Q K^T) must fail the gate, although the
        # mean of V passes the element rule here (|O| ~ 3e-3 < atol).
        with pytest.raises(AssertionError):
            assert_parity(np.zeros_like(got), ref, "all-zero control")
        mean_v = f64(ins[2][0].cuda().float().mean(0))  # [H, D]
        with pytest.raises(AssertionError):
            assert_parity(mean_v[rows % w.H], ref, "mean-of-V control")
