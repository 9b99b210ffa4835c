"""CUDA path vs the fp64 oracle on identical seeded inputs (GPU only).

Tolerance metric (the same everywhere): over all outputs that one test compares,
    err = max |o - o_ref| / max |o_ref|
must be within 1e-5 for fp32 inputs and 1e-2 for bf16 inputs (fp32 accumulation).  The one
shape whose exact output is identically zero is a single token (w_{1,1} = 0, so o_1 = 0; the
fp64 oracle returns rounding noise there): it has no relative error and is held to
max|o - o_ref| <= tolerance in absolute terms, the outputs being built from N(0, 1) values.
Each check also prints the worst ratio of a single (b, h) sequence, for information: a short
sequence can have an output far smaller than the terms of the prefix form that build it (at
two tokens o_2 is proportional to s_1 - s_2 while each term is of the order of the gates), and
there fp32 rounding of those terms, not the kernel, sets the per-sequence ratio.
The logit s, the prefix sum P, the running maximum m and the scaled prefix sum Et = E e^{-m}
must be bit-identical between the forward pass and the token-by-token decode step.
"""
import numpy as np
import pytest
import torch

import oracle
import zeros_inputs as zi

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


@pytest.fixture(scope="module")
def zs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import zero_sum_prefix_gb300 as m
    m.load()
    return m


def seq_err(o, ref):
    """max|o - o_ref| / max|o_ref| over every compared output (o, ref: [S, N, d]); absolute
    error for single-token sequences (exact output 0).  Prints it and the worst single-sequence
    ratio."""
    o = np.asarray(o, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    num = np.abs(o - ref).max()
    if ref.shape[1] == 1:  # a single token: o_1 = 0 exactly
        print(f"max abs error {num:.3e} (single token)")
        return num
    den = np.abs(ref).max()
    assert den > 0.0, "two or more tokens with an all-zero reference"
    per_seq = max(np.abs(o[i] - ref[i]).max() / max(np.abs(ref[i]).max(), np.finfo(float).tiny)
                  for i in range(ref.shape[0]))
    print(f"error {num / den:.3e} (worst single sequence {per_seq:.3e})")
    return num / den


def run(zs, inp, w, **kw):
    return zs.fwd(inp["q"], inp["k"], inp["v"], inp["u"], inp["g1"], inp["gh"], inp["mu"],
                  inp["tau"], causal=w.causal, rope=w.rope, rope_base=w.rope_base, **kw)


def oracle_subset(inp, w, heads, N=None):
    """fp64 oracle outputs for the listed (b, h) sequences: [len(heads), N, d]."""
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])[None]  # noqa: E731
    hs = [h for _, h in heads]
    q, k, v, u = (sel(inp[n]).cpu() for n in ("q", "k", "v", "u"))
    g1, gh = sel(inp["g1"]).cpu(), sel(inp["gh"]).cpu()
    # every sampled sequence keeps its own head's prior: run heads one at a time
    outs = []
    for i, h in enumerate(hs):
        o = oracle.forward(q[:, i:i + 1], k[:, i:i + 1], v[:, i:i + 1], u[:, i:i + 1],
                           g1[:, i:i + 1], gh[:, i:i + 1], inp["mu"][h:h + 1].cpu(),
                           inp["tau"][h:h + 1].cpu(), causal=w.causal, rope=w.rope,
                           rope_base=w.rope_base)
        outs.append(o[0, 0])
    return np.stack(outs)


def gpu_subset(o, heads):
    return torch.stack([o[b, h] for b, h in heads]).float().cpu().numpy()


# ---------------------------------------------------------------------------------------------
def test_causal_f32_small_workload(zs):
    w = zi.CAUSAL_F32_SMALL
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert zs.get_status() == 0
    ref = oracle.forward(*(inp[n].cpu() for n in ("q", "k", "v", "u", "g1", "gh", "mu", "tau")),
                         causal=True)
    assert seq_err(o[0].cpu().numpy(), ref[0]) <= TOL["f32"]


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("N", [1, 2, 37, 300])
@pytest.mark.parametrize("causal,rope", [(True, False), (True, True), (False, False),
                                         (False, True)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_shapes(zs, d, N, causal, rope, dtype):
    w = zi.Workload("small", 2, 3, N, d, dtype=dtype, causal=causal, rope=rope, rope_base=500.0,
                    seed=1000 + N + d)
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert zs.get_status() == 0
    heads = [(b, h) for b in range(2) for h in range(3)]
    ref = oracle_subset(inp, w, heads)
    assert seq_err(gpu_subset(o, heads), ref) <= TOL[dtype]


def test_causal_rope_b8h8n4096d64_full(zs):
    w = zi.CAUSAL_ROPE_B8H8N4096D64
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert zs.get_status() == 0
    assert torch.isfinite(o.float()).all()
    heads = zi.sample_heads(w, 6)
    assert seq_err(gpu_subset(o, heads), oracle_subset(inp, w, heads)) <= TOL["bf16"]


def test_encoder_b256h3n197d64_full(zs):
    w = zi.ENCODER_VIT_B256H3N197D64
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert zs.get_status() == 0
    assert torch.isfinite(o.float()).all()
    heads = zi.sample_heads(w, 24)
    assert seq_err(gpu_subset(o, heads), oracle_subset(inp, w, heads)) <= TOL["bf16"]


def test_long_rope_b2h16n65536d128_full(zs):
    w = zi.LONG_ROPE_B2H16N65536D128
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert zs.get_status() == 0
    assert torch.isfinite(o.float()).all()
    heads = zi.sample_heads(w, 3)
    assert seq_err(gpu_subset(o, heads), oracle_subset(inp, w, heads)) <= TOL["bf16"]


# ---------------------------------------------------------------------------------------------
def _decode_run(zs, w, inp_prefill, steps, device="cuda"):
    """Prefill with the forward pass, then `steps` decode steps.  Returns the decode outputs
    [steps, B, H, d], the debug scalars of every step and the per-step token inputs."""
    st = torch.empty(zs.state_bytes(w.B, w.H, w.d), dtype=torch.uint8, device=device)
    if inp_prefill is not None:
        zs.fwd(inp_prefill["q"], inp_prefill["k"], inp_prefill["v"], inp_prefill["u"],
               inp_prefill["g1"], inp_prefill["gh"], inp_prefill["mu"], inp_prefill["tau"],
               causal=True, rope=w.rope, rope_base=w.rope_base, final_state=st)
    else:
        raise AssertionError("use new_state for an empty prefill")
    outs, dbgs, toks = [], [], []
    for i in range(steps):
        tk = zi.decode_tokens(w, i, device)
        o, dbg = zs.decode_step(st, tk["q"], tk["k"], tk["v"], tk["u"], tk["g1"], tk["gh"],
                                debug=True)
        outs.append(o)
        dbgs.append(dbg)
        toks.append(tk)
    return st, outs, dbgs, toks


@pytest.mark.parametrize("d,rope,dtype", [(32, False, "f32"), (64, True, "bf16"),
                                          (128, True, "bf16"), (128, False, "bf16")])
def test_decode_matches_forward_bitexact(zs, d, rope, dtype):
    """Prefill N0 tokens, decode the rest: s, P, m, Et bit-identical to a forward pass over
    the whole sequence; outputs within tolerance of the oracle."""
    B, H, N0, steps = 2, 3, 45, 20
    w = zi.Workload("dec", B, H, N0, d, dtype=dtype, rope=rope, rope_base=10000.0, seed=77 + d)
    pre = zi.make(w, "cuda")
    st, outs, dbgs, toks = _decode_run(zs, w, pre, steps)
    assert zs.get_status() == 0
    # full sequence = prefill tokens followed by the decoded tokens
    full = {n: torch.cat([pre[n]] + [t[n].unsqueeze(2) for t in toks], dim=2)
            for n in ("q", "k", "v", "u", "g1", "gh")}
    full["mu"], full["tau"] = pre["mu"], pre["tau"]
    wf = w.with_(N=N0 + steps)
    o_full, dbg_full = run(zs, full, wf, debug=True)
    for key in ("s", "E", "P", "m"):
        dec = torch.stack([dg[key] for dg in dbgs], dim=2)  # [B, H, steps]
        fwd = dbg_full[key][:, :, N0:]
        assert torch.equal(dec.view(torch.int32), fwd.contiguous().view(torch.int32)), key
    dec_o = torch.stack(outs, dim=2)  # [B, H, steps, d]
    heads = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle_subset(full, wf, heads)[:, N0:]
    assert seq_err(gpu_subset(dec_o, heads), ref) <= TOL[dtype]
    assert seq_err(gpu_subset(o_full[:, :, N0:], heads), ref) <= TOL[dtype]
    # the state records the token count
    view = zs.state_view(st, B, H, d)
    assert (view["t"] == N0 + steps).all()


@pytest.mark.parametrize("rope", [False, True])
def test_decode_after_long_prefill_d128(zs, rope):
    """The recurrent-decode workload's per-sequence shape: an 8192-token prefill at d = 128 on
    the chunked tensor-core path (as the workload, without RoPE, and with it), then 64 decode
    steps.  Logits and prefix scalars of every step equal those of a forward pass over all 8256
    tokens bit for bit (every sequence); the decode outputs of four seeded (b, h) sequences
    match the fp64 oracle over the whole sequence."""
    base = zi.DECODE_B256H32D128
    steps = 64
    w = base.with_(B=2, H=4, rope=rope)
    N0 = w.N
    pre = zi.make(w, "cuda")
    st, outs, dbgs, toks = _decode_run(zs, w, pre, steps)
    assert zs.get_status() == 0
    full = {n: torch.cat([pre[n]] + [t[n].unsqueeze(2) for t in toks], dim=2)
            for n in ("q", "k", "v", "u", "g1", "gh")}
    full["mu"], full["tau"] = pre["mu"], pre["tau"]
    wf = w.with_(N=N0 + steps)
    _, dbg_full = run(zs, full, wf, debug=True)
    assert zs.get_status() == 0
    for key in ("s", "E", "P", "m"):
        dec = torch.stack([dg[key] for dg in dbgs], dim=2)
        fwd = dbg_full[key][:, :, N0:]
        assert torch.equal(dec.view(torch.int32), fwd.contiguous().view(torch.int32)), key
    heads = zi.sample_heads(w, 4)
    ref = oracle_subset(full, wf, heads)[:, N0:]
    dec_o = torch.stack(outs, dim=2)
    assert seq_err(gpu_subset(dec_o, heads), ref) <= TOL["bf16"]
    view = zs.state_view(st, w.B, w.H, w.d)
    assert (view["t"] == N0 + steps).all()


def test_decode_from_empty_state(zs):
    B, H, d, steps = 3, 2, 64, 24
    w = zi.Workload("dec0", B, H, steps, d, rope=True, seed=91)
    inp = zi.make(w, "cuda")
    st = zs.new_state(inp["mu"], inp["tau"], B, rope=True, rope_base=w.rope_base)
    outs, dbgs = [], []
    for t in range(steps):
        o, dbg = zs.decode_step(st, *(inp[n][:, :, t].contiguous() for n in
                                      ("q", "k", "v", "u", "g1", "gh")), debug=True)
        outs.append(o)
        dbgs.append(dbg)
    o_f, dbg_f = run(zs, inp, w, debug=True)
    for key in ("s", "E", "P", "m"):
        dec = torch.stack([dg[key] for dg in dbgs], dim=2)
        assert torch.equal(dec.view(torch.int32), dbg_f[key].view(torch.int32)), key
    heads = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle_subset(inp, w, heads)
    assert seq_err(gpu_subset(torch.stack(outs, dim=2), heads), ref) <= TOL["bf16"]


def test_decode_header_lookup(zs):
    """zeros_decode_step on a state blob restored into fresh memory reads its header."""
    B, H, d = 2, 2, 32
    w = zi.Workload("hdr", B, H, 10, d, seed=5)
    inp = zi.make(w, "cuda")
    st = torch.empty(zs.state_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    run(zs, inp, w, final_state=st)
    saved = st.cpu()
    restored = saved.cuda()  # a new allocation the library has never seen
    tk = zi.decode_tokens(w, 0, "cuda")
    o1 = zs.decode_step(restored, tk["q"], tk["k"], tk["v"], tk["u"], tk["g1"], tk["gh"])
    o2 = zs.decode_step(st, tk["q"], tk["k"], tk["v"], tk["u"], tk["g1"], tk["gh"])
    assert torch.equal(o1, o2)
    assert torch.equal(restored, st)


def test_device_range_error_is_reported(zs):
    w = zi.Workload("range", 1, 1, 8, 32, dtype="f32", seed=3)
    inp = zi.make(w, "cuda")
    inp["u"][0, 0, 3] = 3.0e38  # the prior-mean numerator overflows -> non-finite logit
    run(zs, inp, w)
    assert zs.get_status() == zs.ZEROS_ERR_RANGE
    assert zs.get_status() == 0  # reading clears it
    inp = zi.make(w, "cuda")
    run(zs, inp, w)
    assert zs.get_status() == 0


def test_empty_and_invalid_calls(zs):
    w = zi.Workload("e", 1, 2, 0, 64, seed=1)
    inp = zi.make(w, "cuda")
    o = run(zs, inp, w)
    assert o.numel() == 0
    q = torch.zeros((1, 1, 4, 48), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((1, 1, 4), dtype=torch.float32, device="cuda")
    mu = torch.zeros((1, 48), dtype=torch.float32, device="cuda")
    tau = torch.zeros((1,), dtype=torch.float32, device="cuda")
    with pytest.raises(zs.ZerosError) as e:
        zs.fwd(q, q, q, q, g, g, mu, tau)
    assert e.value.code == zs.ZEROS_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("rope", [False, True])
def test_chunk_path_small_shapes(zs, d, N, rope):
    """The tcgen05 chunked scan against the oracle (ragged tails, single chunks, many chunks)
    and its logits / prefix sums against the token-sequential path, bit for bit."""
    w = zi.Workload("chunk", 2, 2, N, d, rope=rope, seed=3000 + N + d)
    inp = zi.make(w, "cuda")
    o_c, dbg_c = run(zs, inp, w, path="chunk", debug=True)
    assert zs.get_status() == 0
    o_s, dbg_s = run(zs, inp, w, path="simt", debug=True)
    for key in ("s", "E", "P", "m"):
        assert torch.equal(dbg_c[key].view(torch.int32), dbg_s[key].view(torch.int32)), key
    heads = [(b, h) for b in range(2) for h in range(2)]
    ref = oracle_subset(inp, w, heads)
    assert seq_err(gpu_subset(o_c, heads), ref) <= TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [333, 256, 31, 32, 33])
def test_chunk_final_state_matches_simt(zs, d, N):
    """The prefill state written by the chunked path equals the token-sequential one (scalars
    bit-exact, matrices within bf16-operand rounding)."""
    B, H = 2, 3
    w = zi.Workload("chunkstate", B, H, N, d, rope=True, seed=4242 + d)
    inp = zi.make(w, "cuda")
    st_c = torch.empty(zs.state_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    st_s = torch.empty_like(st_c)
    run(zs, inp, w, path="chunk", final_state=st_c)
    run(zs, inp, w, path="simt", final_state=st_s)
    assert zs.get_status() == 0
    vc, vs = zs.state_view(st_c, B, H, d), zs.state_view(st_s, B, H, d)
    for key in ("t", "mC", "EC", "CP", "etau", "ml", "El", "LP", "C", "L", "mu"):
        assert torch.equal(vc[key], vs[key]), key
    for key in ("F", "G", "H"):
        err = (vc[key] - vs[key]).abs().max() / vs[key].abs().max()
        assert err < 2e-2, (key, float(err))


@pytest.mark.parametrize("d,N", [(64, 4096 + 300), (128, 2 * 2048 + 37)])
def test_chunk_scalars_across_segments_bitexact(zs, d, N):
    """The scalar pass walks a sequence in segments (4096 tokens at d = 64, 2048 at d = 128)
    and carries the column sums and the scalar folds from one segment to the next: the per-token
    logits and prefix scalars, and the scalar part of the prefill state, equal the
    token-sequential path's bit for bit past the segment boundaries (ragged last block)."""
    B, H = 1, 2
    w = zi.Workload("segments", B, H, N, d, rope=True, seed=5151 + d)
    inp = zi.make(w, "cuda")
    st_c = torch.empty(zs.state_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    st_s = torch.empty_like(st_c)
    _, dbg_c = run(zs, inp, w, path="chunk", debug=True, final_state=st_c)
    _, dbg_s = run(zs, inp, w, path="simt", debug=True, final_state=st_s)
    assert zs.get_status() == 0
    for key in ("s", "E", "P", "m"):
        assert torch.equal(dbg_c[key].view(torch.int32), dbg_s[key].view(torch.int32)), key
    vc, vs = zs.state_view(st_c, B, H, d), zs.state_view(st_s, B, H, d)
    for key in ("t", "mC", "EC", "CP", "etau", "ml", "El", "LP", "C", "L", "mu"):
        assert torch.equal(vc[key], vs[key]), key
