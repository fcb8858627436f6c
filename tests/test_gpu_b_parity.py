"""GPU parity: the CUDA forward against the fp64 oracle on the same seeded inputs.

Every call goes through the C ABI (the ctypes binding).  Bar (against the
unrounded oracle): max |out err| <= 2e-2, mean |out err| <= 2e-3,
max |lse err| <= 1e-3.
"""
import numpy as np
import pytest
import torch

from exact_attention_68_gb300 import binding
from exact_attention_68_gb300.workloads import WORKLOADS, check_rows, default_scale, make_qkv
from gpu_helpers import compare, run_gpu, to_f64
from oracle import attention_fwd, attention_rows

pytestmark = pytest.mark.gpu


def _oracle_rows(q, k, v, scale, causal, idx):
    return attention_rows(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal, idx)


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_workload_parity(cuda_device, name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, seed=0)
    scale = default_scale(w.D)
    out, lse = run_gpu(q, k, v, scale, w.causal)
    idx = check_rows(w)
    ro, rl = _oracle_rows(q, k, v, scale, w.causal, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    s = compare(og, lg, ro, rl, name)
    print(name, s)



@pytest.mark.parametrize("S,D", [(4096, 128), (8192, 64)])
def test_ragged_head_groups(cuda_device, S, D):
    """(b, h) slices are scheduled in groups whose K/V fit in L2 (24 slices
    here); 40 slices do not divide into them evenly.  Rows 0, 127, 128, S-1 of
    every slice, every row of the last slice and 512 rows drawn by
    default_rng(3) are compared."""
    B, H = 2, 20
    q, k, v = make_qkv((B, H, S, D), seed=13)
    scale = default_scale(D)
    out, lse = run_gpu(q, k, v, scale, True)
    rows = [(b, h, i) for b in range(B) for h in range(H) for i in (0, 127, 128, S - 1)]
    rows += [(B - 1, H - 1, i) for i in range(S)]
    rng = np.random.default_rng(3)
    rows += [(int(b), int(h), int(i)) for b, h, i in
             zip(rng.integers(0, B, 512), rng.integers(0, H, 512), rng.integers(0, S, 512))]
    idx = np.asarray(rows, dtype=np.int64)
    ro, rl = _oracle_rows(q, k, v, scale, True, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, ro, rl, f"ragged groups S={S} D={D}")

# The persistent kernel brings Q into tensor memory one of two ways, chosen by
# the average K/V steps a tile meets (24 or fewer: through the K ring and
# tcgen05.cp; more: loaded by the softmax warps).  Shapes on both sides of
# that line under each mask: causal averages (n_kt + 1) / 2 steps (S = 6144:
# 24, S = 6272: 25), non-causal n_kt (S = 3072: 24, S = 3200: 25).
Q_PATH_SHAPES = [(6144, True), (6272, True), (3072, False), (3200, False)]


@pytest.mark.parametrize("S,causal", Q_PATH_SHAPES, ids=lambda x: str(x))
@pytest.mark.parametrize("D", [64, 128])
def test_both_q_paths(cuda_device, S, causal, D):
    """Rows 0, 127, 128, S-1 and 256 rows from default_rng(21) of each of the
    three heads against the oracle."""
    B, H = 1, 3
    q, k, v = make_qkv((B, H, S, D), seed=21)
    scale = default_scale(D)
    out, lse = run_gpu(q, k, v, scale, causal)
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([[0, 127, 128, S - 1], rng.integers(0, S, 256)]))
    idx = np.asarray([(0, h, int(i)) for h in range(H) for i in rows], dtype=np.int64)
    ro, rl = _oracle_rows(q, k, v, scale, causal, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, ro, rl, f"S={S} causal={causal} D={D}")


EDGE_SHAPES = [
    (1, 1, 1, 64), (1, 1, 1, 128), (1, 1, 7, 64), (1, 1, 7, 128), (2, 3, 129, 64),
    (1, 2, 200, 128), (1, 1, 256, 128), (1, 1, 384, 64), (3, 1, 1000, 128), (1, 2, 640, 64),
    (2, 1, 513, 128),
]


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_edge_shapes_full_oracle(cuda_device, shape, causal):
    q, k, v = make_qkv(shape, seed=11)
    scale = default_scale(shape[3])
    out, lse = run_gpu(q, k, v, scale, causal)
    ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
    compare(to_f64(out), to_f64(lse), ro, rl, f"{shape} causal={causal}")


@pytest.mark.parametrize("scale", [0.03, 0.5])
@pytest.mark.parametrize("D", [64, 128])
def test_other_scales(cuda_device, scale, D):
    q, k, v = make_qkv((2, 2, 300, D), seed=5, qk_std=2.0)
    for causal in (True, False):
        out, lse = run_gpu(q, k, v, scale, causal)
        ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
        compare(to_f64(out), to_f64(lse), ro, rl, f"scale={scale} D={D} causal={causal}")


def test_peaked_softmax_many_rescales(cuda_device):
    """Large logits whose running max keeps climbing along the keys."""
    q, k, v = make_qkv((1, 4, 1024, 128), seed=6, qk_std=4.0)
    # make later keys larger so the running max moves at many tiles
    ramp = torch.linspace(0.5, 2.0, 1024).view(1, 1, 1024, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    scale = default_scale(128)
    for causal in (True, False):
        out, lse = run_gpu(q, k, v, scale, causal)
        ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
        compare(to_f64(out), to_f64(lse), ro, rl, f"peaked causal={causal}")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_reference_moves_on_every_tile(cuda_device, D):
    """Logits built to climb by about 40 log2 units from each 128-key tile to
    the next, so every row's reference max moves (by more than the bf16
    threshold of 32) on every tile, with the rescale of O and the redo of the
    tile's exponentials each time; the within-tile spread keeps the softmax
    from collapsing onto a single key."""
    S = 1024
    g = torch.Generator().manual_seed(17)
    q = torch.randn(1, 2, S, D, generator=g) * 0.5
    k = torch.randn(1, 2, S, D, generator=g) * 0.5
    v = torch.randn(1, 2, S, D, generator=g)
    scale = default_scale(D)
    # coordinate 0 carries the climb: s_ij gains q_i0 * k_j0 * scale
    q[..., 0] = 4.0
    step = 40.0 / 1.4426950408889634 / (4.0 * scale)  # +40 log2 units per tile
    k[..., 0] = step * (torch.arange(S) // 128).float()
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    for causal in (True, False):
        out, lse = run_gpu(q, k, v, scale, causal)
        ro, rl = attention_fwd(q.float().numpy(), k.float().numpy(), v.float().numpy(), scale, causal)
        compare(to_f64(out), to_f64(lse), ro, rl, f"moving reference D={D} causal={causal}")


def test_constant_v_closed_form(cuda_device):
    """Every V row equal to c gives out = c (rounded to bf16) for every row."""
    q, k, _ = make_qkv((1, 2, 777, 128), seed=8)
    c = torch.linspace(-3, 3, 128).to(torch.bfloat16)
    v = c.view(1, 1, 1, 128).expand(1, 2, 777, 128).contiguous()
    for causal in (True, False):
        out, _ = run_gpu(q, k, v, default_scale(128), causal)
        err = (out.double() - c.double()).abs().max().item()
        assert err <= 2e-2


def test_first_causal_row_is_v0(cuda_device):
    q, k, v = make_qkv((2, 3, 512, 64), seed=9)
    out, lse = run_gpu(q, k, v, default_scale(64), True)
    np.testing.assert_array_equal(out[:, :, 0].float().numpy(), v[:, :, 0].float().numpy())
    ref = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) * default_scale(64)
    assert (lse[:, :, 0].double() - ref).abs().max().item() <= 1e-3


def test_causal_rows_ignore_later_keys_bitwise(cuda_device):
    """Changing K/V rows after i leaves rows <= i bit-identical (c3 shape)."""
    w = WORKLOADS["c3"]
    q, k, v = make_qkv(w, seed=0)
    scale = default_scale(w.D)
    out1, lse1 = run_gpu(q, k, v, scale, True)
    i0 = 1000  # inside a Q tile, so the diagonal tile is partly perturbed
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator().manual_seed(99)
    k2[:, :, i0 + 1:] = torch.randn(k2[:, :, i0 + 1:].shape, generator=g).to(torch.bfloat16)
    v2[:, :, i0 + 1:] = torch.randn(v2[:, :, i0 + 1:].shape, generator=g).to(torch.bfloat16)
    out2, lse2 = run_gpu(q, k2, v2, scale, True)
    assert torch.equal(out1[:, :, :i0 + 1], out2[:, :, :i0 + 1])
    assert torch.equal(lse1[:, :, :i0 + 1], lse2[:, :, :i0 + 1])
    assert not torch.equal(out1[:, :, i0 + 1:], out2[:, :, i0 + 1:])


def test_bitwise_deterministic(cuda_device):
    w = WORKLOADS["c2"]
    q, k, v = make_qkv(w, seed=0)
    a = run_gpu(q, k, v, default_scale(w.D), True)
    b = run_gpu(q, k, v, default_scale(w.D), True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_staged_host_entry_point_matches(cuda_device):
    q, k, v = make_qkv((1, 4, 1024, 128), seed=12)
    scale = default_scale(128)
    ref_out, ref_lse = run_gpu(q, k, v, scale, True)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    out_h = torch.empty_like(q).pin_memory()
    lse_h = torch.empty(ref_lse.shape, dtype=torch.float32).pin_memory()
    dev = torch.device("cuda:0")
    qd, kd, vd = (torch.empty_like(x, device=dev) for x in (q, k, v))
    od = torch.empty_like(qd)
    ld = torch.empty(ref_lse.shape, dtype=torch.float32, device=dev)
    binding.attn_fwd_staged(qh, kh, vh, out_h, lse_h, qd, kd, vd, od, ld, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(out_h, ref_out) and torch.equal(lse_h, ref_lse)


@pytest.mark.parametrize("shape", [(2, 9, 8192, 128), (1, 13, 16384, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_staged_chunked_pipeline_is_bitwise_the_device_path(cuda_device, shape):
    """Inputs large enough that the staged call splits the slices into chunks
    (18 slices into 3 even chunks; 13 into 7 + 6) whose copies and kernels
    overlap on internal streams; two calls back to back on the same buffers,
    each followed by a kernel on the caller's stream that reads the device
    output, must see that call's own result."""
    scale = default_scale(shape[3])
    dev = torch.device("cuda:0")
    q1, k1, v1 = make_qkv(shape, seed=14)
    q2, k2, v2 = make_qkv(shape, seed=15)
    refs = [run_gpu(q, k, v, scale, True) for q, k, v in ((q1, k1, v1), (q2, k2, v2))]
    hosts = [tuple(x.pin_memory() for x in t) for t in ((q1, k1, v1), (q2, k2, v2))]
    outs = [torch.empty_like(q1).pin_memory() for _ in range(2)]
    lses = [torch.empty(shape[:3], dtype=torch.float32).pin_memory() for _ in range(2)]
    qd, kd, vd = (torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(3))
    od = torch.empty_like(qd)
    ld = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    sums = []
    for n in range(2):
        binding.attn_fwd_staged(*hosts[n], outs[n], lses[n], qd, kd, vd, od, ld, scale=scale,
                                causal=True)
        sums.append(od.float().sum())  # a kernel on the caller's stream after the call
    torch.cuda.synchronize()
    assert binding.device_status() == binding.ATTN_OK
    for n in range(2):
        assert torch.equal(outs[n], refs[n][0]) and torch.equal(lses[n], refs[n][1])
        # the same reduction on the GPU over the reference output: bitwise equal
        assert sums[n].item() == refs[n][0].to(dev).float().sum().item()


def test_binding_rejects_wrong_dtype_and_layout(cuda_device):
    q, k, v = (x.to("cuda:0") for x in make_qkv((1, 1, 128, 64)))
    with pytest.raises(TypeError):
        binding.attn_fwd(q.float(), k, v)
    with pytest.raises(ValueError):
        binding.attn_fwd(q.transpose(1, 2), k, v)
    with pytest.raises(binding.AttnError):
        binding.attn_fwd(q, k, v, scale=-1.0)


def test_binding_rejects_outputs_of_the_wrong_size_type_or_device(cuda_device):
    """Every buffer the library writes or copies must be exactly the size,
    type and side (host or device) the call implies: checked in the binding
    before anything is enqueued."""
    shape = (1, 2, 128, 64)
    q, k, v = (x.to("cuda:0") for x in make_qkv(shape))
    out, lse = binding.attn_fwd(q, k, v)
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, out=torch.empty(shape, dtype=torch.bfloat16))  # host out
    with pytest.raises(ValueError):
        binding.attn_fwd(q, k, v, lse=torch.empty(shape[:3]))                     # host lse
    dout = torch.ones_like(q)
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, out, lse, dout, dq=torch.empty(shape, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        binding.attn_bwd(q, k, v, out, lse, dout, delta=torch.empty(shape[:3]))
    with pytest.raises(ValueError):
        binding.attn_fwd_noalloc(q, k, v, torch.empty(shape, dtype=torch.bfloat16), lse)
    hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
    hout = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(shape[:3]).pin_memory()
    dq_, dk_, dv_ = (torch.empty_like(q) for _ in range(3))
    dout_, dlse_ = torch.empty_like(q), torch.empty_like(lse)
    small = torch.empty((1, 1, 128, 64), dtype=torch.bfloat16).pin_memory()
    for bad in ({"q_h": small}, {"out_h": small}, {"lse_h": torch.empty((1, 2, 64))},
                {"q_h": hq.float()}, {"out_d": dout_[:, :1]}, {"lse_d": dlse_.cpu()}):
        kw = dict(q_h=hq, k_h=hk, v_h=hv, out_h=hout, lse_h=hlse, q_d=dq_, k_d=dk_, v_d=dv_,
                  out_d=dout_, lse_d=dlse_)
        kw.update(bad)
        with pytest.raises(ValueError):
            binding.attn_fwd_staged(**kw)
    # the valid call still works and matches the device path
    binding.attn_fwd_staged(hq, hk, hv, hout, hlse, dq_, dk_, dv_, dout_, dlse_)
    torch.cuda.synchronize()
    assert torch.equal(hout, out.cpu()) and torch.equal(hlse, lse.cpu())


@pytest.mark.parametrize("D", [64, 128])
def test_long_context_131072(cuda_device, D):
    """The longest context here: S = 131072 (1024 Q tiles, 512 units of the
    causal triangle per slice).  Rows 0, 1, 127, 128, S/2, S-129, S-1 and 48
    rows from default_rng(7) of each of the two heads against the oracle."""
    B, H, S = 1, 2, 131072
    q, k, v = make_qkv((B, H, S, D), seed=16)
    scale = default_scale(D)
    out, lse = run_gpu(q, k, v, scale, True)
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, S // 2, S - 129, S - 1], rng.integers(0, S, 48)]))
    idx = np.asarray([(0, h, int(i)) for h in range(H) for i in rows], dtype=np.int64)
    ro, rl = _oracle_rows(q, k, v, scale, True, idx)
    og = to_f64(out)[idx[:, 0], idx[:, 1], idx[:, 2]]
    lg = to_f64(lse)[idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(og, lg, ro, rl, f"S=131072 D={D}")
