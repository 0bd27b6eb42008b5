"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by
element, within max abs 2e-3 and relative L2 1e-3 on the fp32 output.

Small cases span several 32-token tiles, several 512-token partitions and ragged tails,
for every format, head size and group size built; the described workloads run at full size
in the benchmark's launch configuration and are compared with the oracle on their whole
output."""
import math

import numpy as np
import pytest
import torch

from decode_attention_paged_gqa_gb300 import workloads as wl
from paged_cases import assert_close, make_case, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

EDGE_LENS = [0, 1, 15, 16, 17, 511, 512, 513, 1023, 1024, 1025, 1500, 2053]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from decode_attention_paged_gqa_gb300 import build

    build.build()


def small_spec(fmt, D, G, Hkv=2, window=0, softcap=0.0, lens=EDGE_LENS, seed=7):
    spec = wl.WorkloadSpec(f"edge_{fmt}_{D}_{G}", len(lens), Hkv * G, Hkv, D, fmt, 0, max(lens), seed=seed,
                           window=window, softcap=softcap)
    return spec, wl.make_layout(spec, lens=lens)


def test_tiny_bf16_unsplit_and_split():
    spec = wl.WORKLOADS["tiny_bf16"]
    c = make_case(spec)
    ref = run_oracle(c)
    assert_close(run_gpu(c, partition_size=0), ref, "tiny unsplit")
    assert_close(run_gpu(c, partition_size=512, split_threshold=1024), ref, "tiny split (2 partitions)")
    assert_close(run_gpu(c, partition_size=512, split_threshold=1), ref, "tiny split forced")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_edge_lengths(fmt, D, G):
    spec, lay = small_spec(fmt, D, G, seed=D + G)
    c = make_case(spec, lay)
    assert_close(run_gpu(c), run_oracle(c), f"{fmt} D{D} G{G}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("window,softcap", [(100, 0.0), (1000, 0.0), (1024, 30.0), (0, 5.0), (4096, 50.0)])
def test_window_and_softcap(fmt, window, softcap):
    spec, lay = small_spec(fmt, 128, 4, window=window, softcap=softcap, lens=EDGE_LENS + [4097, 5000], seed=window)
    c = make_case(spec, lay)
    assert_close(run_gpu(c), run_oracle(c), f"{fmt} window={window} softcap={softcap}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("schedule", [1, 2])
@pytest.mark.parametrize("D,G,T,window", [(128, 4, 1, 0), (256, 2, 1, 700), (128, 2, 3, 0), (128, 8, 1, 0),
                                          (128, 4, 4, 300)])
def test_partition_schedules(fmt, schedule, D, G, T, window):
    """Both ways of dealing a CTA's partitions to its warps (shared by the warps, or each warp
    owning whole partitions), with the automatic and with three partitions per CTA (rounded up
    to the warps when they own partitions), unsplit and split sequences, windows, multi-token
    queries and eight columns."""
    lens = [0, 1, 17, 1023, 1024, 1500, 2053, 4097, 5000, 9000]
    spec = wl.WorkloadSpec(f"sched_{fmt}", len(lens), 2 * G, 2, D, fmt, 0, max(lens), seed=31 + D + G + T,
                           window=window, query_len=T)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    ref = run_oracle(c)
    for ppc in (0, 3):
        assert_close(run_gpu(c, partition_schedule=schedule, partitions_per_cta=ppc), ref,
                     f"{fmt} schedule {schedule}, {ppc} partitions per CTA")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("T,window,softcap,schedule", [(1, 0, 0.0, 0), (1, 700, 30.0, 2), (2, 0, 0.0, 1),
                                                       (3, 0, 0.0, 2)])
def test_alibi(fmt, T, window, softcap, schedule):
    """ALiBi slopes (one per query head, the usual geometric choice), with one and several
    query tokens, a window and softcap, under both partition schedules."""
    lens = [1, 17, 600, 1030, 2500, 4100]
    G = 2
    spec = wl.WorkloadSpec(f"alibi_{fmt}", len(lens), 4 * G, 4, 128, fmt, 0, max(lens), seed=50 + T + window,
                           window=window, softcap=softcap, query_len=T)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / 8) for h in range(8)], np.float32)
    gpu = run_gpu(c, alibi_slopes=torch.from_numpy(slopes).cuda(), partition_schedule=schedule)
    assert_close(gpu, run_oracle(c, alibi_slopes=slopes), f"{fmt} alibi T{T} W{window} cap{softcap}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("placement", ["k_below_v", "v_below_k", "one_buffer"])
def test_cache_placement(fmt, placement):
    """The kernels fetch a page of K and of V (and of their norms) with one copy through a
    map spanning both arrays when it can, whichever lies lower in memory, and with one copy
    per array otherwise (here: K and V given as the same buffer, so the values are the keys)."""
    spec, lay = small_spec(fmt, 128, 4, lens=[5, 600, 1500, 2100], seed=61)
    c = make_case(spec, lay)
    dev = to_device(c)
    if placement == "one_buffer":
        if c["k"].shape != c["v"].shape or c["k"].dtype != c["v"].dtype:
            pytest.skip("K and V rows differ in size for this format")
        c = dict(c, v=c["k"], v_scales=c["k_scales"])
        dev["v"], dev["v_scales"] = dev["k"], dev["k_scales"]
    else:
        def pair(k, v):  # both in one allocation, in the requested order, 256-byte aligned
            nk = (k.numel() * k.element_size() + 255) // 256 * 256
            nv = (v.numel() * v.element_size() + 255) // 256 * 256
            buf = torch.empty(nk + nv, dtype=torch.uint8, device="cuda")
            lo, hi = (buf[:nk], buf[nk:]) if placement == "k_below_v" else (buf[nv:], buf[:nv])
            k2 = lo[:k.numel() * k.element_size()].view(k.dtype).view(k.shape)
            v2 = hi[:v.numel() * v.element_size()].view(v.dtype).view(v.shape)
            k2.copy_(k)
            v2.copy_(v)
            return k2, v2
        dev["k"], dev["v"] = pair(dev["k"], dev["v"])
        if dev["k_scales"] is not None and dev["k_scales"].numel() > 1:
            dev["k_scales"], dev["v_scales"] = pair(dev["k_scales"], dev["v_scales"])
    assert_close(run_gpu(c, dev=dev), run_oracle(c), f"{fmt} {placement}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "cb3k_cb4v"])
@pytest.mark.parametrize("schedule", [1, 2])
def test_back_to_back_calls_see_fresh_inputs(fmt, schedule):
    """Calls queued back to back on one stream, sharing one workspace, with the query and the
    context lengths rewritten by stream-ordered copies between them and no host sync: each
    phase is launched early (programmatic dependent launch) and must still read what the
    copies and the previous call left, and each call's partials must not mix with the next's."""
    import decode_attention_paged_gqa_gb300 as da
    from paged_cases import params_for

    lens = [0, 17, 1023, 1500, 2053, 4097]
    spec = wl.WorkloadSpec(f"b2b_{fmt}", len(lens), 8, 2, 128, fmt, 0, max(lens), seed=77)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    dev = to_device(c)
    p = params_for(c, partition_schedule=schedule)
    ws = torch.empty(da.decode_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    da.decode_attn_workspace_init(p)
    variants = []
    for i in range(4):
        q_i = torch.roll(c["q"], shifts=i, dims=-2)  # heads rotated: every output row changes
        lens_i = np.maximum(c["lens"] - 301 * i, 0).astype(c["lens"].dtype)
        variants.append((q_i, lens_i))
    q_src = [q.cuda() for q, _ in variants]
    len_src = [torch.from_numpy(ln).cuda() for _, ln in variants]
    outs = [torch.full(tuple(c["q"].shape), float("nan"), dtype=torch.float32, device="cuda") for _ in variants]
    torch.cuda.synchronize()
    for i in range(len(variants)):
        dev["q"].copy_(q_src[i])
        dev["lens"].copy_(len_src[i])
        da.decode_attn_paged(dev["q"], dev["k"], dev["v"], dev["k_scales"], dev["v_scales"], dev["codebook"],
                             dev["sign"], dev["bt"], dev["lens"], outs[i], p)
    torch.cuda.synchronize()
    assert da.decode_attn_get_device_error(p) == 0
    for i, (q_i, lens_i) in enumerate(variants):
        assert_close(outs[i].cpu().numpy(), run_oracle(dict(c, q=q_i, lens=lens_i)), f"{fmt} call {i}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4"])
def test_cuda_graph_capture_and_replay(fmt):
    """decode_attn_paged captured into a CUDA graph (its phases launched with programmatic
    stream serialisation become graph nodes) and replayed with new query contents gives the
    oracle's result on every replay."""
    import decode_attention_paged_gqa_gb300 as da
    from paged_cases import params_for

    lens = [0, 17, 1500, 4097]
    spec = wl.WorkloadSpec(f"graph_{fmt}", len(lens), 8, 2, 128, fmt, 0, max(lens), seed=91)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    dev = to_device(c)
    p = params_for(c)
    ws = torch.empty(da.decode_attn_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    da.attach_workspace(p, ws)
    da.decode_attn_workspace_init(p)
    out = torch.full(tuple(c["q"].shape), float("nan"), dtype=torch.float32, device="cuda")

    def call():
        da.decode_attn_paged(dev["q"], dev["k"], dev["v"], dev["k_scales"], dev["v_scales"], dev["codebook"],
                             dev["sign"], dev["bt"], dev["lens"], out, p)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one call outside the capture: the launchers' one-time set-up
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for i in range(3):
        q_i = torch.roll(c["q"], shifts=i + 1, dims=-2)
        dev["q"].copy_(q_i.cuda())
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), run_oracle(dict(c, q=q_i)), f"{fmt} replay {i}")
    assert da.decode_attn_get_device_error(p) == 0


@pytest.mark.parametrize("fmt", ["bf16", "cb4"])
def test_maximum_partition_count(fmt):
    """The largest grid the library takes: 8192 partitions of 16 tokens for a 131072-token
    sequence (the reduce then combines 8192 partials per row), next to a ragged shorter one."""
    lens = [131072, 70001]
    spec = wl.WorkloadSpec(f"maxp_{fmt}", len(lens), 8, 2, 128, fmt, 0, max(lens), seed=123)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    ref = run_oracle(c, partition_size=0)
    assert_close(run_gpu(c, partition_size=16, split_threshold=1), ref, f"{fmt}, 8192 partitions")


@pytest.mark.parametrize("psize,thresh", [(0, 1024), (16, 1), (48, 64), (512, 1), (4096, 1024)])
def test_partition_sizes(psize, thresh):
    spec, lay = small_spec("bf16", 128, 4, lens=EDGE_LENS, seed=psize + 3)
    c = make_case(spec, lay)
    ref = run_oracle(c, partition_size=0)
    assert_close(run_gpu(c, partition_size=psize, split_threshold=thresh), ref, f"psize {psize}")


@pytest.mark.parametrize("name", ["llama3_8b_bf16", "fp8_long_32k", "gemma_window_softcap", "cb4_long_32k",
                                  "fp8k_cb4v_long_32k", "cb3k_cb4v_long_32k"])
def test_full_size_workloads_whole_output(name):
    """The described workloads at full size, in the benchmark's launch configuration: every
    (sequence, head) row of the output against the oracle, max abs elementwise and relative
    L2 over the whole [B, Hq, D] tensor."""
    spec = wl.WORKLOADS[name]
    c = make_case(spec)
    out = run_gpu(c)
    ref = run_oracle(c)
    assert out.shape == ref.shape == (spec.batch, spec.num_q_heads, spec.head_dim)
    max_abs, rel = assert_close(out, ref, name)
    print(f"{name}: whole output, max_abs={max_abs:.3e} rel_l2={rel:.3e}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
def test_spread_context_lengths(fmt):
    """A batch whose context lengths spread from 1 to 32768 tokens (unsplit and split sequences,
    1 to 64 partitions each) in the automatic launch configuration: the codebook-value kernel
    deals this uneven work to its warps from one flattened list of items."""
    lens = [1, 32768, 17, 300, 20000, 1023, 1024, 7000, 2500, 12345, 512, 4097, 31999, 64]
    spec = wl.WorkloadSpec(f"spread_{fmt}", len(lens), 32, 8, 128, fmt, 0, max(lens), seed=404)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    assert_close(run_gpu(c), run_oracle(c), f"{fmt} spread lengths")


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
@pytest.mark.parametrize("B,T,window", [(16, 1, 0), (16, 2, 0), (48, 1, 2048)])
def test_small_batch_one_wave(fmt, B, T, window):
    """Small batches of spread lengths (1 to 8192 tokens) whose partitions, at the longest
    possible span, fill at least two waves of the tensor-core kernel's CTAs but few enough
    that every sequence's partitions fit one wave in chunks of at most 8: the kernel then runs
    one wave and picks the chunk size from the lengths in-kernel. Each partition's partial does
    not depend on how partitions are chunked, so the output must equal, bit for bit, that of
    the fixed grid of one partition per CTA; and it must match the oracle."""
    rng = np.random.default_rng(1000 + B + T)
    lens = [int(x) for x in rng.integers(1, 8193, size=B)]
    lens[:6] = [1, 512, 513, 1024, 1025, 8192]
    spec = wl.WorkloadSpec(f"wave_{fmt}", B, 32, 8, 128, fmt, 0, 8192, seed=77 + B, window=window, query_len=T)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    dev = to_device(c)
    auto = run_gpu(c, dev)
    fixed = run_gpu(c, dev, partition_schedule=1, partitions_per_cta=1)
    np.testing.assert_array_equal(auto, fixed)
    assert_close(auto, run_oracle(c), f"{fmt} B={B} T={T} window={window} one wave")


@pytest.mark.parametrize("fmt", ["bf16", "fp8"])
@pytest.mark.parametrize("qscale", [1e-3, 3e2, 1e5])
def test_query_magnitudes(fmt, qscale):
    """The FP8 path computes q.k with f16 operands: queries far outside the f16 range must
    still give the right answer (they are rescaled by a power of two, exactly)."""
    spec, lay = small_spec(fmt, 128, 4, lens=[1, 600, 1500], seed=11)
    c = make_case(spec, lay)
    c["q"] = (c["q"].float() * qscale).to(torch.bfloat16)
    assert_close(run_gpu(c, softmax_scale=1.0 / (qscale * math.sqrt(128))), run_oracle(
        c, softmax_scale=1.0 / (qscale * math.sqrt(128))), f"{fmt} q x{qscale}")


@pytest.mark.parametrize("fmt", ["fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("vscale", [1e-30, 3e4])
def test_value_magnitudes(fmt, vscale):
    """Value scales far from 1: the 4-bit value side multiplies P by the token's norm before a
    16-bit MMA, which must neither overflow (norms ~3e5 here, above the f16 range) nor lose
    tiny norms."""
    spec, lay = small_spec(fmt, 128, 4, lens=[1, 600, 1500], seed=13)
    c = make_case(spec, lay)
    c["v_scales"] = c["v_scales"] * vscale
    ref = run_oracle(c)
    scale = float(np.abs(ref).max())
    assert_close(run_gpu(c) / scale, ref / scale, f"{fmt} v x{vscale}")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "cb3k_cb4v"])
def test_rising_scores(fmt):
    """Scores that rise slowly along the context (about one log2 unit per page) keep the
    lazily moved softmax reference stale for many pages before it moves."""
    lens = [16 * 40 + 5, 2500]
    spec, lay = small_spec(fmt, 128, 4, lens=lens, seed=17)
    q_dir = torch.zeros(128)
    q_dir[0] = 1.0
    nb = lay.num_blocks
    k = torch.randn(nb, 2, 16, 128) * 0.05
    # key of (block, slot) at token position t gets a component along q's first axis that
    # grows with t: block_tables map positions to blocks, so walk them
    for b, L in enumerate(lens):
        for t in range(L):
            phys = int(lay.block_tables[b, t // 16])
            k[phys, :, t % 16, 0] = t / 16.0
    c = make_case(spec, lay, sources={"k": k})
    q = torch.zeros_like(c["q"].float())
    q[..., 0] = 8.0
    c["q"] = q.to(torch.bfloat16)
    assert_close(run_gpu(c), run_oracle(c), f"{fmt} rising scores")


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "cb4", "fp8k_cb4v", "cb3k_cb4v"])
@pytest.mark.parametrize("T,G,window", [(2, 4, 0), (4, 2, 0), (3, 2, 700), (8, 1, 0), (2, 1, 1000), (5, 1, 64),
                                        (4, 4, 0), (8, 4, 0), (4, 8, 0), (3, 4, 900), (5, 4, 0), (32, 1, 0)])
def test_multi_token_causal(fmt, T, G, window):
    """T query tokens per sequence at positions L-T .. L-1, each attending positions up to its
    own (multi-token / speculative decode). More than 8 (query token, head) pairs are split
    into column groups of 8, one CTA each (T * G up to 32)."""
    lens = [3, 17, 600, 1024, 1030, 2500]  # includes fewer tokens than queries
    spec = wl.WorkloadSpec(f"mt_{fmt}", len(lens), 2 * G, 2, 128, fmt, 0, max(lens), seed=T * 10 + G, window=window,
                           query_len=T)
    c = make_case(spec, wl.make_layout(spec, lens=lens))
    out = run_gpu(c)
    assert out.shape == (len(lens), T, 2 * G, 128)
    assert_close(out, run_oracle(c), f"{fmt} T{T} G{G} W{window}")


def test_multi_token_group_too_wide_is_rejected():
    import decode_attention_paged_gqa_gb300 as da

    spec = wl.WorkloadSpec("wide", 2, 8, 2, 128, "bf16", 10, 40, seed=1, query_len=9)  # 9 x 4 > 32
    c = make_case(spec)
    with pytest.raises(da.DecodeAttnError) as e:
        run_gpu(c)
    assert e.value.status == da._binding.DA_ERR_UNSUPPORTED
