"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Criterion (the pages' UT/ATK metric): per output,
RMS(gpu - oracle) / RMS(oracle) < 1e-3, with the output dtype exact; qk_dot's
indexing/layout is checked bit-exactly with marker inputs.  The oracle runs
in BF16-boundary mode.  Small problems compare every element; the full-size
workloads compare every output element of sampled (b, h) heads.
"""

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.gpu
TOL = 1e-3
DTYPES = {"dmimo_o": torch.float32, "states": torch.bfloat16, "dz": torch.bfloat16,
          "dmimo_z": torch.float32, "qk_dot": torch.bfloat16}


def rel_rms(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.sqrt(np.mean(b ** 2))
    num = np.sqrt(np.mean((a - b) ** 2))
    return float(num / den) if den > 0 else float(num)


def to_dev(inp, dev="cuda"):
    return [a.to(dev) if isinstance(a, torch.Tensor) else a for a in si.args_of(inp)]


def run_gpu(inp):
    out = mm.mamba_mimo_bwd_fwd(*to_dev(inp))
    torch.cuda.synchronize()
    return out


def compare(got, want, tag=""):
    errs = {}
    for name in oracle.OUTPUT_NAMES:
        g, w = getattr(got, name), want[name]
        assert (g is None) == (w is None), (tag, name)
        if g is None:
            continue
        assert g.dtype == DTYPES[name], (tag, name, g.dtype)
        gn = g.float().cpu().numpy()
        assert gn.shape == w.shape, (tag, name, gn.shape, w.shape)
        assert np.all(np.isfinite(gn)), (tag, name, "non-finite values")
        errs[name] = rel_rms(gn, w)
    bad = {k: v for k, v in errs.items() if not v < TOL}
    assert not bad, f"{tag}: rel-RMS over {TOL}: {bad} (all: {errs})"
    return errs


def check(inp, tag=""):
    got = run_gpu(inp)
    want = oracle.bwd_fwd(*si.args_of(inp))
    return compare(got, want, tag)


def unit_inputs(seed=123, batch=1, seqlen=32, heads=1, groups=1, state_dim=64, value_dim=64,
                rank=4, chunk_size=16, reduce_o=True, has_z=False, has_d=False, div=4,
                recipe="unit"):
    return si.make_inputs(B=batch, S=seqlen, H=heads, G=groups, R=rank, N=state_dim, P=value_dim,
                          C=chunk_size, div=div, reduced=reduce_o, has_z=has_z, has_d=has_d,
                          seed=seed, recipe=recipe)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


# --- the pages' unit-test matrix (PR #125 test file), both value recipes ----

@pytest.mark.parametrize("recipe", ["unit", "workload"])
@pytest.mark.parametrize("reduce_o,has_z,has_d", [(True, False, False), (True, True, True),
                                                   (False, False, True), (False, True, False)])
def test_branches(recipe, reduce_o, has_z, has_d):
    check(unit_inputs(reduce_o=reduce_o, has_z=has_z, has_d=has_d, recipe=recipe))


def test_gqa():
    check(unit_inputs(heads=2, groups=1, has_z=True, has_d=True))


@pytest.mark.parametrize("seed", [0, 1, 42])
def test_tail_seeds(seed):
    check(unit_inputs(seed=seed, seqlen=35, heads=2, has_z=True, has_d=True))


def test_batch_groups():
    check(unit_inputs(batch=2, heads=4, groups=2, seqlen=20, has_z=True, has_d=True))


def test_non_power_of_two_tail():
    check(unit_inputs(seqlen=13, rank=3, chunk_size=6, has_z=True, has_d=True))


def test_tail_chunk():
    check(unit_inputs(seqlen=20, has_z=True, has_d=True))


@pytest.mark.parametrize("N,P,R,C", [(32, 64, 4, 16), (128, 32, 4, 16), (64, 128, 4, 16),
                                     (128, 64, 8, 8), (64, 64, 3, 6), (64, 64, 1, 64)])
def test_shapes(N, P, R, C):
    check(unit_inputs(seqlen=2 * C, state_dim=N, value_dim=P, rank=R, chunk_size=C))


# --- edge cases of the envelope ----------------------------------------------

@pytest.mark.parametrize("kw", [
    dict(seqlen=1, chunk_size=1, rank=1, state_dim=2, value_dim=1, div=2),      # smallest
    dict(seqlen=5, chunk_size=1, rank=2, state_dim=4, value_dim=3),             # C = 1
    dict(seqlen=300, chunk_size=128, rank=1, state_dim=128, value_dim=128, div=2),  # C*R = 128, max N/P
    dict(seqlen=64, chunk_size=16, rank=8, state_dim=128, value_dim=128),       # C*R = 128, R = 8
    dict(seqlen=40, chunk_size=8, rank=16, state_dim=16, value_dim=20),         # R = 16
    dict(seqlen=37, chunk_size=5, rank=3, state_dim=12, value_dim=5, div=2),    # odd P, N not /16
    dict(seqlen=50, chunk_size=7, rank=2, state_dim=20, value_dim=33, heads=3, groups=3),
    dict(seqlen=17, chunk_size=16, rank=4, state_dim=8, value_dim=130 - 2),     # two p-slices
    # shapes of the specialised kernels, with tails and GQA
    dict(seqlen=200, chunk_size=16, rank=4, state_dim=64, value_dim=64, heads=4, groups=2),
    dict(seqlen=77, chunk_size=16, rank=8, state_dim=64, value_dim=64, heads=2, groups=1),
    dict(seqlen=90, chunk_size=16, rank=4, state_dim=32, value_dim=32, heads=3, groups=1),
])
@pytest.mark.parametrize("branches", [(True, True, True), (False, True, False), (True, False, True)])
def test_edge_shapes(kw, branches):
    r, z, d = branches
    check(unit_inputs(reduce_o=r, has_z=z, has_d=d, recipe="workload", **kw), str(kw))


# --- the synthetic workloads -------------------------------------------------

@pytest.mark.parametrize("index", [0, 1])
def test_small_workloads_full(index):
    check(si.workload_inputs(index), si.WORKLOADS[index].name)


def sampled_heads(index, pairs):
    """Full-size workload on the GPU (inputs drawn on the device), every output
    element of the sampled (b, h) heads compared with the oracle run on those
    heads' input slices."""
    wl = si.WORKLOADS[index]
    inp = si.make_inputs(**wl.shape_kwargs(), seed=si.WORKLOAD_SEED_BASE + index, device="cuda")
    got = mm.mamba_mimo_bwd_fwd(*si.args_of(inp))
    torch.cuda.synchronize()
    variant = mm.last_kernel_variant()
    if index in (2, 3, 4):   # shapes with specialised kernels must use them
        assert variant >= 0, f"{wl.name} ran the generic kernels"
    if index == 2:        # the timed shape runs the warp-specialised tensor-core kernel
        assert variant == 3, f"{wl.name} ran kernel family {variant}"
    if index == 3:        # the wide-state family (256-byte N rows, C*R = 128)
        assert variant == 4, f"{wl.name} ran kernel family {variant}"
    for (b, h) in pairs:
        sl = si.head_slice(inp, b, h)
        sl_cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in sl.items()}
        want = oracle.bwd_fwd(*si.args_of(sl_cpu))
        head = mm.MambaMimoBwdFwdOutputs(
            None if got.dmimo_o is None else got.dmimo_o[b:b + 1, h:h + 1],
            got.states[b:b + 1, h:h + 1],
            None if got.dz is None else got.dz[b:b + 1, :, h:h + 1],
            None if got.dmimo_z is None else got.dmimo_z[b:b + 1, h:h + 1],
            got.qk_dot[b:b + 1, h:h + 1])
        compare(head, want, f"{wl.name} head ({b},{h})")
    del inp, got
    torch.cuda.empty_cache()


def test_timed_workload_all_heads():
    # every output element of all 16 heads of the pages' timed shape, in the
    # benchmark's launch configuration (the oracle runs all heads at once)
    wl = si.WORKLOADS[2]
    inp = si.make_inputs(**wl.shape_kwargs(), seed=si.WORKLOAD_SEED_BASE + 2, device="cuda")
    got = mm.mamba_mimo_bwd_fwd(*si.args_of(inp))
    torch.cuda.synchronize()
    assert mm.last_kernel_variant() == 3 and mm.last_plan()["single_kernel"] == 1
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    want = oracle.bwd_fwd(*si.args_of(cpu))
    compare(got, want, wl.name)
    del inp, got
    torch.cuda.empty_cache()


def test_wide_state_workload_sampled_heads():
    sampled_heads(3, [(0, 0), (1, 31)])


def test_throughput_workload_sampled_heads():
    sampled_heads(4, [(0, 3), (7, 31)])


# --- layout, determinism, coverage -------------------------------------------

@pytest.mark.parametrize("C,R,N,P,S", [(8, 4, 8, 8, 19), (16, 4, 64, 64, 37), (16, 8, 64, 64, 21)])
def test_qk_dot_layout_bit_exact(C, R, N, P, S):
    # q[t,r] = (2^(8r + 16 (t%2) - 60), 0, ...), k[t,s] = (2^s, 0, ...), biases 0:
    # every same-token product is a distinct power of two, exact in BF16.
    inp = unit_inputs(seqlen=S, chunk_size=C, rank=R, state_dim=N, value_dim=P, recipe="workload")
    q = torch.zeros_like(inp["q"])
    k = torch.zeros_like(inp["k"])
    for t in range(S):
        for r in range(R):
            q[0, t, r, 0, 0] = 2.0 ** (8 * r + 16 * (t % 2) - 60)
            k[0, t, r, 0, 0] = 2.0 ** r
    inp.update(q=q, k=k, q_bias=torch.zeros_like(inp["q_bias"]), k_bias=torch.zeros_like(inp["k_bias"]))
    got = run_gpu(inp).qk_dot.float().cpu()
    want = torch.tensor(oracle.bwd_fwd(*si.args_of(inp))["qk_dot"], dtype=torch.float32)
    assert torch.equal(got, want)
    assert got[0, 0, 3, 2, 1] == 2.0 ** (8 * 2 + 16 - 60 + 1)


def test_deterministic_and_every_output_written():
    inp = si.workload_inputs(1)
    a = run_gpu(inp)
    # second call into NaN-filled outputs: every element must be overwritten
    nan_out = mm.MambaMimoBwdFwdOutputs(*[None if t is None else torch.full_like(t, float("nan"))
                                          for t in a])
    b = mm.mamba_mimo_bwd_fwd(*to_dev(inp), out=nan_out)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        if x is not None:
            assert torch.equal(x, y)


def test_all_outputs_written_with_z_and_reduced():
    inp = si.workload_inputs(0)
    ref = run_gpu(inp)
    nan_out = mm.MambaMimoBwdFwdOutputs(*[torch.full_like(t, float("nan")) for t in ref])
    b = mm.mamba_mimo_bwd_fwd(*to_dev(inp), out=nan_out)
    torch.cuda.synchronize()
    for x, y in zip(ref, b):
        assert torch.equal(x, y)


def test_launch_count_reported():
    run_gpu(si.workload_inputs(0))
    assert mm.last_launch_count() >= 2


def test_device_status_clean_after_calls():
    # every wait inside the kernels is bounded; a completed call reports no timeout
    for index in (0, 1):
        run_gpu(si.workload_inputs(index))
        mm.device_status()
    wl = si.WORKLOADS[2]
    inp = si.make_inputs(**wl.shape_kwargs(), seed=7, device="cuda")
    mm.mamba_mimo_bwd_fwd(*si.args_of(inp))
    assert mm.last_kernel_variant() == 3
    mm.device_status()


# --- inputs outside the workload ranges --------------------------------------

# one case per kernel family: the warp-specialised tensor-core kernel (R4 C16
# N=P=64, reduced dout), the specialised kernels with per-rank dout, R = 8,
# N = P = 32, and the generic kernels
FAMILIES = [
    dict(seqlen=70, heads=2, reduce_o=True, has_z=True, has_d=True),
    dict(seqlen=70, heads=2, reduce_o=False, has_z=True, has_d=True),
    dict(seqlen=45, heads=2, rank=8, reduce_o=True, has_z=True, has_d=True),
    dict(seqlen=50, heads=2, state_dim=32, value_dim=32, reduce_o=True, has_z=True, has_d=True),
    dict(seqlen=37, heads=2, rank=3, chunk_size=6, state_dim=24, value_dim=20, reduce_o=True, has_z=True,
         has_d=True),
]


def poison_segsum(inp):
    """+inf and NaN on and above the diagonal of every segsum block: entries
    the strictly causal mask excludes.  The mask must be a select, so none of
    them may reach an output (a mask applied by multiplication would turn
    them into NaN)."""
    seg = inp["segsum"].clone()
    C = seg.shape[-1]
    i = torch.arange(C)
    upper = i[None, :] >= i[:, None]
    pattern = torch.where((i[None, :] + i[:, None]) % 2 == 0, torch.tensor(float("inf")),
                          torch.tensor(float("nan")))
    seg[..., upper] = pattern[upper]
    out = dict(inp)
    out["segsum"] = seg
    return out


@pytest.mark.parametrize("kw", FAMILIES)
def test_segsum_inf_nan_above_diagonal(kw):
    inp = poison_segsum(unit_inputs(recipe="workload", **kw))
    assert torch.isnan(inp["segsum"]).any() and torch.isposinf(inp["segsum"]).any()
    check(inp, str(kw))


@pytest.mark.parametrize("kw", FAMILIES)
def test_large_rotary_angles(kw):
    # rotary angles of real models reach the thousands; the specialised
    # kernels reduce them by 2 pi before sin.approx / cos.approx
    inp = unit_inputs(recipe="workload", **kw)
    g = torch.Generator().manual_seed(2024)
    inp["angles"] = (torch.rand(inp["angles"].shape, generator=g, dtype=torch.float64) * 4e4 - 2e4).float()
    check(inp, str(kw))


def test_workspace_size_independent_of_device():
    # The launch plan is a function of the problem only: the size queried with
    # a GPU current equals the size queried in a process that sees no GPU, so a
    # workspace sized anywhere is accepted by every call.
    import json
    import os
    import subprocess
    import sys
    shapes = [(1, 8192, 16, 1, 4, 64, 64, 16, 4, 1, 1), (2, 16384, 32, 4, 4, 128, 64, 32, 2, 1, 1),
              (8, 32768, 32, 8, 8, 64, 64, 16, 4, 1, 1), (2, 1000, 8, 2, 4, 32, 32, 16, 4, 0, 0),
              (1, 200, 2, 1, 4, 64, 64, 16, 4, 0, 1)]
    code = (
        "import ctypes, json, sys; sys.path.insert(0, %r)\n"
        "import mamba_mimo_chunked_gb300 as mm\n"
        "lib = mm.load_library(); out = []\n"
        "for B, S, H, G, R, N, P, C, div, red, z in %r:\n"
        "    d = mm._Dims(B, S, H, G, R, N, P); n = ctypes.c_size_t(0)\n"
        "    assert lib.mamba_mimo_bwd_fwd_workspace_size(ctypes.byref(d), C, div, red, z, ctypes.byref(n)) == 0\n"
        "    out.append(n.value)\n"
        "print(json.dumps(out))\n") % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))), shapes)
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    no_gpu = json.loads(subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                                       check=True).stdout)
    here = []
    for B, S, H, G, R, N, P, C, div, red, z in shapes:
        here.append(mm.workspace_size(B, S, H, G, R, N, P, C, div, bool(red), bool(z)))
    assert here == no_gpu


# --- both forms of the warp-specialised tensor-core family -------------------

@pytest.mark.parametrize("two_kernel", [False, True])
@pytest.mark.parametrize("kw", [
    dict(seqlen=200, heads=2, has_z=True, has_d=True),                  # several segments
    dict(seqlen=1000, heads=3, groups=1, has_z=True, has_d=False),      # ragged tail
    dict(seqlen=64, batch=2, heads=4, groups=2, has_z=False, has_d=True),
    dict(seqlen=16, heads=1, has_z=True, has_d=True),                   # one chunk
    dict(seqlen=2005, heads=16, has_z=True, has_d=True),                # 14-chunk segments, ragged tail
    dict(seqlen=3000, batch=2, heads=8, groups=2, has_z=True, has_d=True),  # 21 / 20-chunk segments, GQA
])
def test_tensor_core_family_forms(kw, two_kernel):
    lib = mm.load_library()
    lib.mamba_mimo_set_test_hooks(2 if two_kernel else 0)
    try:
        inp = unit_inputs(recipe="workload", **kw)
        got = run_gpu(inp)
        assert mm.last_kernel_variant() == 3
        assert mm.last_plan()["single_kernel"] == (0 if two_kernel else 1)
        assert mm.last_launch_count() == (2 if two_kernel else 1)
    finally:
        lib.mamba_mimo_set_test_hooks(0)
    compare(got, oracle.bwd_fwd(*si.args_of(inp)), str(kw))


def test_timed_workload_two_kernel_form_sampled_heads():
    lib = mm.load_library()
    lib.mamba_mimo_set_test_hooks(2)
    try:
        sampled_heads(2, [(0, 0), (0, 9)])
        assert mm.last_plan()["single_kernel"] == 0
    finally:
        lib.mamba_mimo_set_test_hooks(0)


# --- the wide-state family: R4 C32 N=128 P=64, rotary on all of N -------------

@pytest.mark.parametrize("branches", [(True, True, True), (True, False, False), (False, True, True),
                                      (False, False, True)])
@pytest.mark.parametrize("kw", [
    dict(seqlen=200, heads=2),                         # ragged tail, several segments
    dict(seqlen=1000, batch=2, heads=4, groups=2),     # GQA, B = 2, multi-segment prefix
    dict(seqlen=32, heads=1),                          # one full chunk
    dict(seqlen=5, heads=1),                           # one partial chunk
])
def test_wide_state_family(kw, branches):
    r, z, d = branches
    inp = unit_inputs(state_dim=128, value_dim=64, rank=4, chunk_size=32, div=2, reduce_o=r, has_z=z,
                      has_d=d, recipe="workload", **kw)
    got = run_gpu(inp)
    # per-rank dout is a [C*R][P] stage tile the wide family has no room for:
    # those calls run the generic kernels
    assert mm.last_kernel_variant() == (4 if r else -1)
    compare(got, oracle.bwd_fwd(*si.args_of(inp)), f"{kw} {branches}")
