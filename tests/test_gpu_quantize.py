"""GPU parity of the MXFP8 quantizer against the CPU oracle: bit-exact codes and scales
("End-to-End MXFP8 RL on Blackwell", section "The pipeline", paragraph "The format";
column-wise copies: the learner paragraph; sync-path equality: section "The grid, byte
for byte")."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from mxfp8_block_scaled_05_gb300 import workloads as W
from tests.oracle_helpers import bf16_bits, bits_to_bf16, gpu_ready, load_golden, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def m():
    mod = gpu_ready()
    yield mod
    assert mod.device_status() == mod.OK


def _expect_scales(rs, layout):
    return rs.reshape(-1) if layout == O.LINEAR else O.swizzle_scales(rs)


def _check(m, x_bf16_cpu, axis, layout):
    q, s = m.quantize(x_bf16_cpu.to(DEV), axis, layout)
    rq, rs = O.quantize(bf16_bits(x_bf16_cpu), axis)
    np.testing.assert_array_equal(u8(q), rq)
    np.testing.assert_array_equal(u8(s).reshape(-1), _expect_scales(rs, layout))


@pytest.mark.parametrize("axis", [O.ROW, O.COL])
@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_tiny_config(m, axis, layout):
    a, w = W.tiny("cpu", seed=0)
    _check(m, a, axis, layout)
    _check(m, w, axis, layout)


def _rand_bf16(g, shape, spread=True):
    x = g.standard_normal(shape)
    if spread:
        x *= np.exp2(g.integers(-30, 30, size=(shape[0], 1)))
    f = x.astype(np.float32).view(np.uint32)
    return bits_to_bf16(((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16))


@pytest.mark.parametrize("shape", [(1, 32), (33, 96), (160, 160), (255, 4128), (129, 32), (384, 640)])
@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_row_ragged_shapes(m, shape, layout):
    _check(m, _rand_bf16(np.random.default_rng(sum(shape)), shape), O.ROW, layout)


@pytest.mark.parametrize("shape", [(32, 8), (64, 24), (160, 136), (288, 264), (4096, 40), (96, 1000)])
@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_col_ragged_shapes(m, shape, layout):
    _check(m, _rand_bf16(np.random.default_rng(sum(shape) + 1), shape), O.COL, layout)


@pytest.mark.parametrize("context", [0x0000, 0x3F80, 0x7180], ids=["alone", "beside1", "beside2^100"])
def test_brute_force_every_bf16(m, context):
    """Every BF16 bit pattern (NaN and Inf included) in element 0 of a block whose
    element 1 is 0, 1.0 or 2^100; row-wise and column-wise."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = np.zeros((65536, 32), np.uint16)
    x[:, 0] = allb
    x[:, 1] = context
    _check(m, bits_to_bf16(x), O.ROW, O.LINEAR)
    _check(m, bits_to_bf16(np.ascontiguousarray(x.T)), O.COL, O.LINEAR)


def test_hand_worked_blocks(m):
    """The hand-derived golden blocks, straight against the fixture."""
    cases = load_golden("hand_blocks.json")["blocks"]
    nb = (len(cases) + 7) // 8 * 8            # column-wise needs cols % 8 == 0: pad with zero blocks
    x = np.zeros((nb, 32), np.uint16)
    want = np.zeros((nb, 32), np.uint8)
    want_s = np.zeros(nb, np.uint8)
    for i, c in enumerate(cases):
        for j, h in enumerate(c["bf16"]):
            x[i, j] = int(h, 16)
        want[i] = int(c.get("fill_code", "0x00"), 16)
        for j, h in enumerate(c["codes"]):
            want[i, j] = int(h, 16)
        want_s[i] = int(c["scale"], 16)
    q, s = m.quantize(bits_to_bf16(x).to(DEV), m.ROW, m.LINEAR)
    np.testing.assert_array_equal(u8(q), want)
    np.testing.assert_array_equal(u8(s)[:, 0], want_s)
    # the same blocks along the token dimension
    q, s = m.quantize(bits_to_bf16(np.ascontiguousarray(x.T)).to(DEV), m.COL, m.LINEAR)
    np.testing.assert_array_equal(u8(q), want)
    np.testing.assert_array_equal(u8(s)[:, 0], want_s)


def test_empty_and_invariants(m):
    q, s = m.quantize(torch.empty((0, 64), dtype=torch.bfloat16, device=DEV), m.ROW, m.SWIZZLED)
    assert q.numel() == 0 and s.numel() == 0
    x = _rand_bf16(np.random.default_rng(3), (256, 512))
    q, s = m.quantize(x.to(DEV), m.ROW, m.LINEAR)
    codes, scales = u8(q), u8(s)
    assert not np.any((codes & 0x7F) == 0x7F)                     # finite codes only
    # quantize(dequantize(q)) == q: dequantized with torch's float8 view (exact in BF16
    # for these exponents) and re-quantized on the GPU
    deq = (q.view(torch.float8_e4m3fn).float().view(256, 16, 32)
           * torch.exp2(s.float() - 127.0)[..., None]).view(256, 512).to(torch.bfloat16)
    q2, s2 = m.quantize(deq, m.ROW, m.LINEAR)
    assert torch.equal(q2, q) and torch.equal(s2, s)
    np.testing.assert_array_equal(codes >> 7, np.signbit(O.bf16_to_f64(bf16_bits(x))).astype(np.uint8))


@pytest.mark.parametrize("axis", [O.ROW, O.COL])
@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_batched_equals_per_item(m, axis, layout):
    g = np.random.default_rng(5)
    xs = torch.stack([_rand_bf16(g, (160, 96)) for _ in range(3)])
    q, s = m.quantize_batched(xs.to(DEV), axis, layout)
    per = m.scale_bytes(160, 96, axis, layout)
    for i in range(3):
        rq, rs = O.quantize(bf16_bits(xs[i]), axis)
        np.testing.assert_array_equal(u8(q[i]), rq)
        np.testing.assert_array_equal(u8(s[i * per:(i + 1) * per]), _expect_scales(rs, layout))


@pytest.mark.parametrize("axis", [O.ROW, O.COL])
def test_grouped_segments(m, axis):
    """Expert segments with empty experts, sizes below / above / at 128, ragged tails."""
    counts = [64, 0, 160, 32, 0, 256, 96, 0]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total = int(off[-1])
    x = _rand_bf16(np.random.default_rng(7), (total, 224))
    offs = torch.from_numpy(off).to(DEV)
    q, s = m.quantize_grouped(x.to(DEV), offs, axis)
    rq, rs = O.quantize(bf16_bits(x), axis)
    np.testing.assert_array_equal(u8(q), rq)
    want = O.swizzle_grouped_rows(rs, off) if axis == O.ROW else O.swizzle_grouped_cols(rs, off)
    np.testing.assert_array_equal(u8(s)[:want.size], want)
    assert m.device_status() == m.OK


def test_grouped_bad_offsets_latched(m):
    """Offsets that are not 32-aligned are refused by the kernel itself: it writes nothing
    and latches MXFP8_ERR_BAD_OFFSETS."""
    x = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([0, 40, 128], dtype=torch.int32, device=DEV)
    out = torch.full((128, 64), 0xAB, dtype=torch.uint8, device=DEV)
    sc = torch.full((m.grouped_scale_bytes(128, 64, 2, m.ROW),), 0xCD, dtype=torch.uint8, device=DEV)
    m.quantize_grouped(x, offs, m.ROW, out=out, scales=sc)
    assert m.device_status() == m.ERR_BAD_OFFSETS
    assert torch.all(out == 0xAB) and torch.all(sc == 0xCD)
    assert m.device_status() == m.OK


def test_status_latched_on_another_stream_is_read_once(m):
    """An error latched by a kernel on one stream is returned by a status read on another
    stream once that kernel has finished, then cleared. The read takes the word with one
    atomic exchange, so every host thread's read gets a status of its own: four threads
    reading at once after one latch see the error exactly once."""
    import threading
    x = torch.zeros((128, 64), dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([0, 40, 128], dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        m.quantize_grouped(x, offs, m.ROW, stream=side)
    side.synchronize()
    assert m.device_status() == m.ERR_BAD_OFFSETS     # read on the default stream
    assert m.device_status() == m.OK
    for _ in range(3):
        with torch.cuda.stream(side):
            m.quantize_grouped(x, offs, m.ROW, stream=side)
        side.synchronize()
        seen = []
        gate = threading.Barrier(4)

        def read():
            s = torch.cuda.Stream()
            gate.wait()
            seen.append(m.device_status(stream=s))

        ts = [threading.Thread(target=read) for _ in range(4)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        assert sorted(seen) == [m.OK] * 3 + [m.ERR_BAD_OFFSETS], seen


def _sample_rows_check(m, x_dev, axis, n_samples, seed):
    """Full-size quantize on the GPU; the oracle recomputes sampled rows (ROW) or sampled
    columns (COL) of the input and both codes and swizzled scale bytes are compared."""
    rows, cols = x_dev.shape
    q, s = m.quantize(x_dev, axis, m.SWIZZLED)
    g = np.random.default_rng(seed)
    if axis == m.ROW:
        idx = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, n_samples)]))
        xb = bf16_bits(x_dev[torch.from_numpy(idx).to(DEV)])
        rq, rs = O.quantize(xb, O.ROW)
        s_cols = cols // 32
    else:
        idx = np.unique(np.concatenate([[0, cols - 1], g.integers(0, cols, n_samples)]))
        xb = bf16_bits(x_dev[:, torch.from_numpy(idx).to(DEV)])
        rq, rs = O.quantize(xb, O.COL)
        s_cols = rows // 32
    np.testing.assert_array_equal(u8(q[torch.from_numpy(idx).to(DEV)]), rq)
    r, c = np.meshgrid(idx, np.arange(s_cols), indexing="ij")
    offs = O.swizzle_offset(r, c, s_cols)
    np.testing.assert_array_equal(u8(s)[offs], rs)
    return q, s


def test_qwen3_8b_layer_set_full_size_sampled(m):
    """Config: Qwen3-8B linears at 4096 tokens; X, W, dY quantized row- and column-wise
    at full size, sampled rows/columns checked bit for bit."""
    for name, n, k, x, w, dy in W.qwen3_8b_layer_set(4096, DEV, seed=1):
        for t in (x, w, dy):
            for axis in (m.ROW, m.COL):
                _sample_rows_check(m, t, axis, 24, seed=n + k + axis)
        del x, w, dy
    torch.cuda.empty_cache()


def test_weight_sync_pass_byte_equality(m):
    """Config: the weight-synchronization pass of a Qwen3-8B-shaped model (36 layers x 4
    projections, 6.95 G elements). Section "The grid, byte for byte": the synced weights
    must be the forward GEMM's weight quantization byte for byte. The two come from
    different kernel paths here:
      - the sync call is mxfp8_quantize (ROW, swizzled scales): the register-tile
        row-wise kernel;
      - the forward operand is the row-wise copy that the forward step makes with
        mxfp8_quantize_dual_multi, the weight quantized in one launch beside its layer's
        activations: the shared-tile dual kernel (the bench step's own call).
    Every one of the 144 weights is compared in full, codes and scales, so a single
    diverging byte between the two row passes fails the test. One weight of each of the
    four shapes is also compared in full with the oracle, and sharded sync calls (row
    shards at 128-row multiples, column shards at 128-column multiples) equal the whole."""
    shapes = W.sync_weight_shapes()
    assert len(shapes) == 144
    g = torch.Generator(device=DEV).manual_seed(40)
    xs = {k: W.activations_bf16(4096, k, g, DEV, 0.005, 30.0) for k in (4096, 12288)}
    total, oracle_checked = 0, set()
    for i, (layer, name, n, k) in enumerate(shapes):
        wt = W.sync_weight(layer, name, n, k, DEV)
        total += wt.numel()
        q_s, s_s = m.quantize(wt, m.ROW, m.SWIZZLED)                   # sync path
        _, (q_f, s_f, _, _) = m.quantize_dual_multi([xs[k], wt], m.SWIZZLED)  # forward path
        assert q_f.data_ptr() != q_s.data_ptr()
        assert torch.equal(q_f, q_s) and torch.equal(s_f, s_s), (layer, name)
        if name not in oracle_checked:
            rq, rs = O.quantize(bf16_bits(wt), O.ROW)
            np.testing.assert_array_equal(u8(q_s), rq)
            np.testing.assert_array_equal(u8(s_s), O.swizzle_scales(rs))
            oracle_checked.add(name)
        if i % 37 == 0:
            # sharded sync: two row shards (128-multiple split) and two column shards
            cut = (n // 2) // 128 * 128
            qa, sa = m.quantize(wt[:cut].contiguous(), m.ROW, m.SWIZZLED)
            qb, sb = m.quantize(wt[cut:].contiguous(), m.ROW, m.SWIZZLED)
            assert torch.equal(torch.cat([qa, qb]), q_f)
            assert torch.equal(torch.cat([sa, sb]), s_f)
            kc = (k // 2) // 128 * 128
            ql, sl = m.quantize(wt[:, :kc].contiguous(), m.ROW, m.LINEAR)
            qr, sr = m.quantize(wt[:, kc:].contiguous(), m.ROW, m.LINEAR)
            q_lin, s_lin = m.quantize(wt, m.ROW, m.LINEAR)
            assert torch.equal(torch.cat([ql, qr], dim=1), q_lin)
            assert torch.equal(torch.cat([sl, sr], dim=1), s_lin)
        del wt, q_f, s_f, q_s, s_s
    assert oracle_checked == {"qkv_proj", "o_proj", "gate_up_proj", "down_proj"}
    assert total == 36 * (6144 * 4096 + 4096 * 4096 + 24576 * 4096 + 4096 * 12288)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", [(32, 32), (160, 96), (4096, 40 * 32), (288, 4128), (4096, 4096),
                                   (4128, 3872)])
@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_dual_equals_both_axes(m, shape, layout):
    """One read, both copies: identical to the oracle's row-wise and column-wise bytes. The
    two large shapes have more 128 x 128 tiles than resident CTAs, so their last wave runs
    as 32-row strips (4128 rows: the last tile row has one strip of data and three of
    padding, whose scale entries must still be zero)."""
    x = _rand_bf16(np.random.default_rng(shape[0] + shape[1]), shape)
    rq, rs, cq, cs = m.quantize_dual(x.to(DEV), layout)
    orq, ors = O.quantize(bf16_bits(x), O.ROW)
    ocq, ocs = O.quantize(bf16_bits(x), O.COL)
    np.testing.assert_array_equal(u8(rq), orq)
    np.testing.assert_array_equal(u8(rs).reshape(-1), _expect_scales(ors, layout))
    np.testing.assert_array_equal(u8(cq), ocq)
    np.testing.assert_array_equal(u8(cs).reshape(-1), _expect_scales(ocs, layout))


@pytest.mark.parametrize("offset", [16, 48])
def test_dual_row_codes_at_16_byte_offsets(m, offset):
    """The row-wise codes leave in 32-byte stores when their buffer is 32-byte aligned and
    in 16-byte stores otherwise: the same oracle bytes at a 16-byte but not 32-byte aligned
    address, with the bytes around the output untouched."""
    shape = (160, 4128)
    x = _rand_bf16(np.random.default_rng(offset), shape)
    n = shape[0] * shape[1]
    buf = torch.full((n + 2 * offset,), 0xA5, dtype=torch.uint8, device=DEV)
    row_out = buf[offset:offset + n].view(shape)
    assert row_out.data_ptr() % 32 == 16
    rq, rs, cq, cs = m.quantize_dual(x.to(DEV), O.SWIZZLED, row_out=row_out)
    orq, ors = O.quantize(bf16_bits(x), O.ROW)
    ocq, ocs = O.quantize(bf16_bits(x), O.COL)
    np.testing.assert_array_equal(u8(rq), orq)
    np.testing.assert_array_equal(u8(cq), ocq)
    np.testing.assert_array_equal(u8(rs).reshape(-1), _expect_scales(ors, O.SWIZZLED))
    np.testing.assert_array_equal(u8(cs).reshape(-1), _expect_scales(ocs, O.SWIZZLED))
    rest = u8(buf)
    assert np.all(rest[:offset] == 0xA5) and np.all(rest[offset + n:] == 0xA5)


@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
def test_multi_job_launch_equals_separate_calls(m, layout):
    """Several tensors in one launch: the oracle's bytes for a small job, and byte equality
    with one quantize_dual per job for ragged shapes, a large one and an empty one."""
    g = np.random.default_rng(23 + layout)
    shapes = [(160, 96), (4096, 4096), (288, 4128), (0, 64), (6144, 4096), (32, 32),
              (96, 4064), (4128, 160)]           # the maximum of 8 jobs per launch
    xs = [_rand_bf16(g, sh).to(DEV) if sh[0] else torch.empty(sh, dtype=torch.bfloat16, device=DEV)
          for sh in shapes]
    got = m.quantize_dual_multi(xs, layout)
    assert m.device_status() == m.OK
    for x, (rq, rs, cq, cs) in zip(xs, got):
        if x.numel() == 0:
            continue
        want = m.quantize_dual(x, layout)
        for a, b in zip((rq, rs, cq, cs), want):
            assert torch.equal(a, b)
    x0 = xs[0].cpu()
    orq, ors = O.quantize(bf16_bits(x0), O.ROW)
    ocq, ocs = O.quantize(bf16_bits(x0), O.COL)
    rq, rs, cq, cs = got[0]
    np.testing.assert_array_equal(u8(rq), orq)
    np.testing.assert_array_equal(u8(rs).reshape(-1), _expect_scales(ors, layout))
    np.testing.assert_array_equal(u8(cq), ocq)
    np.testing.assert_array_equal(u8(cs).reshape(-1), _expect_scales(ocs, layout))


def test_grouped_dual_equals_grouped(m):
    counts = [64, 0, 160, 32, 0, 256, 96, 0]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = _rand_bf16(np.random.default_rng(17), (int(off[-1]), 192))
    offs = torch.from_numpy(off).to(DEV)
    rq, rs, cq, cs = m.quantize_grouped_dual(x.to(DEV), offs)
    orq, ors = O.quantize(bf16_bits(x), O.ROW)
    ocq, ocs = O.quantize(bf16_bits(x), O.COL)
    np.testing.assert_array_equal(u8(rq), orq)
    np.testing.assert_array_equal(u8(cq), ocq)
    want_r = O.swizzle_grouped_rows(ors, off)
    want_c = O.swizzle_grouped_cols(ocs, off)
    np.testing.assert_array_equal(u8(rs)[:want_r.size], want_r)
    np.testing.assert_array_equal(u8(cs)[:want_c.size], want_c)
    assert m.device_status() == m.OK


@pytest.mark.parametrize("context", [0x0000, 0x3F80, 0x7180], ids=["alone", "beside1", "beside2^100"])
def test_round_up_rule_brute_force_every_bf16(m, context):
    """The round-up (never saturating) power-of-two rule, every BF16 value, both axes."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = np.zeros((65536, 32), np.uint16)
    x[:, 0] = allb
    x[:, 1] = context
    for axis, xs in ((O.ROW, x), (O.COL, np.ascontiguousarray(x.T))):
        q, s = m.quantize(bits_to_bf16(xs).to(DEV), axis, m.LINEAR, rule=m.RULE_CEIL)
        rq, rs = O.quantize(xs, axis, rule=O.RULE_CEIL)
        np.testing.assert_array_equal(u8(q), rq)
        np.testing.assert_array_equal(u8(s), rs)


def test_round_up_rule_golden_blocks_and_grid_difference(m):
    cases = load_golden("hand_blocks_ceil.json")["blocks"]
    x = np.zeros((len(cases), 32), np.uint16)
    want = np.zeros((len(cases), 32), np.uint8)
    for i, c in enumerate(cases):
        for j, h in enumerate(c["bf16"]):
            x[i, j] = int(h, 16)
        for j, h in enumerate(c["codes"]):
            want[i, j] = int(h, 16)
    q, s = m.quantize(bits_to_bf16(x).to(DEV), m.ROW, m.LINEAR, rule=m.RULE_CEIL)
    np.testing.assert_array_equal(u8(q), want)
    np.testing.assert_array_equal(u8(s)[:, 0], [int(c["scale"], 16) for c in cases])
    # two grids on one weight: they differ exactly in the blocks whose amax exceeds
    # 448 * 2^e_floor, where the round-up scale byte is one higher
    w = W.sync_weight(0, "o_proj", 4096, 4096, DEV)
    qf, sf = m.quantize(w, m.ROW, m.LINEAR)
    qc, sc = m.quantize(w, m.ROW, m.LINEAR, rule=m.RULE_CEIL)
    amax = w.float().abs().view(4096, 128, 32).amax(dim=2).double().cpu().numpy()
    ef = u8(sf).astype(np.int64) - 127
    over = amax > np.ldexp(448.0, ef)
    diff = u8(sc).astype(np.int64) - u8(sf).astype(np.int64)
    bad = np.argwhere(diff != over.astype(np.int64))
    assert bad.size == 0, (bad[:3], amax[tuple(bad[0])], ef[tuple(bad[0])], diff[tuple(bad[0])])
    blocks_differ = (u8(qf).reshape(4096, 128, 32) != u8(qc).reshape(4096, 128, 32)).any(axis=2)
    assert not np.any(blocks_differ & ~over)
    assert 0.01 < over.mean() < 0.9


def test_largest_token_grid(m):
    """The largest input the quantizer's grid takes: 65535 tiles of 128 token rows (8388480
    rows) x 32 columns, row-wise, column-wise and dual. Sampled rows and columns (every
    token of those columns) against the oracle, first and last ones included."""
    rows, cols = 65535 * 128, 32
    g = torch.Generator(device=DEV).manual_seed(12)
    x = (torch.randn((rows, cols), generator=g, device=DEV) *
         torch.exp2(torch.randint(-20, 20, (rows, 1), generator=g, device=DEV).float())
         ).to(torch.bfloat16)
    from tests.oracle_helpers import check_quantized_sampled
    qr, sr = m.quantize(x, m.ROW, m.SWIZZLED)
    check_quantized_sampled(x, qr, sr, O.ROW, 64, seed=1)
    qc, sc = m.quantize(x, m.COL, m.SWIZZLED)
    check_quantized_sampled(x, qc, sc, O.COL, 2, seed=2)
    dr, dsr, dc, dsc = m.quantize_dual(x, m.SWIZZLED)
    assert torch.equal(dr, qr) and torch.equal(dsr, sr)
    assert torch.equal(dc, qc) and torch.equal(dsc, sc)
    assert m.device_status() == m.OK
    del x, qr, sr, qc, sc, dr, dsr, dc, dsc
    torch.cuda.empty_cache()
