"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each expected value comes from
a fixture written by hand from the code table, a second formulation of the
table, a closed form, a balanced-ternary identity, or a library matmul.
"""
import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def table_from_golden():
    return {int(bits, 2): int(v) for bits, v in read_golden("code_table.txt")}


def second_formulation(packed):
    """The table as the 7B write-up states it in §2.2: sign = (code==1) - (code==2),
    fields read at shifts 0,2,4,6 (low bits first)."""
    b = packed.astype(np.int16)[..., None]
    codes = (b >> np.array([0, 2, 4, 6])) & 3
    t = (codes == 1).astype(np.int8) - (codes == 2).astype(np.int8)
    return t.reshape(packed.shape[0], packed.shape[1] * 4)


def test_code_table(oracle_mod):
    table = table_from_golden()
    assert sorted(table) == [0, 1, 2, 3]
    for code, v in table.items():
        assert oracle_mod.trit(code) == v


def test_byte_0x1a_reads_low_bits_first(oracle_mod):
    (row,) = read_golden("byte_0x1a.txt")
    byte = int(row[0], 16)
    want = [int(v) for v in row[1:]]
    t, reserved = oracle_mod.unpack(np.array([[byte]], dtype=np.uint8))
    assert t[0].tolist() == want
    assert reserved == 0


def test_all_256_bytes_against_second_formulation(oracle_mod):
    packed = np.arange(256, dtype=np.uint8).reshape(256, 1)
    t, reserved = oracle_mod.unpack(packed)
    assert np.array_equal(t, second_formulation(packed))
    # every byte with a field equal to 11: count fields by brute force
    want_reserved = sum(((b >> s) & 3) == 3 for b in range(256) for s in (0, 2, 4, 6))
    assert reserved == want_reserved == 256 * 4 // 4


def test_all_256_bytes_against_golden_table(oracle_mod):
    table = table_from_golden()
    packed = np.arange(256, dtype=np.uint8).reshape(256, 1)
    t, _ = oracle_mod.unpack(packed)
    for b in range(256):
        want = [table[(b >> (2 * j)) & 3] for j in range(4)]
        assert t[b].tolist() == want, hex(b)


def test_unpack_wider_row_field_positions(oracle_mod):
    # one non-zero field per row, at every position of a 3-byte row: catches a
    # wrong byte index or field order
    K = 12
    for k in range(K):
        for code, v in ((1, 1), (2, -1)):
            packed = np.zeros((1, K // 4), dtype=np.uint8)
            packed[0, k // 4] = code << (2 * (k % 4))
            t, _ = oracle_mod.unpack(packed)
            want = np.zeros(K, dtype=np.int8)
            want[k] = v
            assert np.array_equal(t[0], want)


def test_pack_roundtrip_random(oracle_mod):
    rng = np.random.default_rng(1)
    t = rng.integers(-1, 2, size=(37, 64), dtype=np.int8)
    packed, invalid = oracle_mod.pack(t)
    assert invalid == 0
    back, reserved = oracle_mod.unpack(packed)
    assert reserved == 0
    assert np.array_equal(back, t)
    # and the packed bytes agree with the second formulation
    assert np.array_equal(second_formulation(packed), t)


def test_pack_of_unpack_canonicalises_reserved(oracle_mod):
    packed = np.arange(256, dtype=np.uint8).reshape(256, 1)
    t, _ = oracle_mod.unpack(packed)
    again, invalid = oracle_mod.pack(t)
    assert invalid == 0
    # 11 fields become 00; every other field is unchanged
    canon = packed.copy()
    for b in range(256):
        c = b
        for j in range(4):
            if ((b >> (2 * j)) & 3) == 3:
                c &= ~(3 << (2 * j)) & 0xFF
        canon[b, 0] = c
    assert np.array_equal(again, canon)


def test_pack_counts_invalid(oracle_mod):
    t = np.array([[0, 1, -1, 2, 5, -3, 0, 0]], dtype=np.int8)
    packed, invalid = oracle_mod.pack(t)
    assert invalid == 3
    assert packed[0].tolist() == [0b00_10_01_00 | 0, 0]  # invalid entries written as 00


def test_hand_example(oracle_mod):
    rows = read_golden("linear_hand_example.txt")
    packed = np.array([[int(v, 16) for v in r[1:]] for r in rows if r[0] == "packed"],
                      dtype=np.uint8)
    x = np.array([[float(v) for v in r[1:]] for r in rows if r[0] == "x"])
    kv = {r[0]: r[1:] for r in rows if r[0] not in ("packed", "x")}
    s_ch = np.array([float(v) for v in kv["channel_scale"]])
    y_ch = np.array([float(v) for v in kv["channel_y"]]).reshape(2, 2)
    G = int(kv["group_size"][0])
    s_g = np.array([float(v) for v in kv["group_scale"]]).reshape(2, -1)
    y_g = np.array([float(v) for v in kv["group_y"]]).reshape(2, 2)
    assert np.array_equal(oracle_mod.linear_f64(x, packed, s_ch, 0), y_ch)
    assert np.array_equal(oracle_mod.linear_f64(x, packed, s_g, G), y_g)


def test_brute_force_every_byte_balanced_ternary(oracle_mod):
    """Row n = byte n, K=4, x = (1,3,9,27), s = 1: y[n] is the balanced-ternary
    number whose digits are the row's four values, so it identifies them."""
    packed = np.arange(256, dtype=np.uint8).reshape(256, 1)
    x = np.array([[1.0, 3.0, 9.0, 27.0]])
    y = oracle_mod.linear_f64(x, packed, np.ones(256), 0)[0]
    table = table_from_golden()
    for b in range(256):
        digits = [table[(b >> (2 * j)) & 3] for j in range(4)]
        assert y[b] == sum(d * 3 ** j for j, d in enumerate(digits))
    # distinct digit vectors give distinct values: decode back
    for b in range(256):
        v, got = int(y[b]), []
        for _ in range(4):
            r = ((v + 1) % 3) - 1
            got.append(r)
            v = (v - r) // 3
        assert got == [table[(b >> (2 * j)) & 3] for j in range(4)]


@pytest.mark.parametrize("group_size", [0, 128])
def test_closed_forms(oracle_mod, group_size):
    rng = np.random.default_rng(7)
    M, K = 3, 256
    x = rng.standard_normal((M, K))
    groups = K // 128
    rows = {
        "plus": 0x55,   # every field 01
        "minus": 0xAA,  # every field 10
        "zero": 0x00,
        "reserved": 0xFF,
    }
    packed = np.stack([np.full(K // 4, v, dtype=np.uint8) for v in rows.values()])
    N = packed.shape[0]
    if group_size == 0:
        s = np.array([0.5, 0.25, 3.0, 7.0])
        y = oracle_mod.linear_f64(x, packed, s, 0)
        np.testing.assert_allclose(y[:, 0], 0.5 * x.sum(1), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(y[:, 1], -0.25 * x.sum(1), rtol=1e-13, atol=1e-13)
    else:
        s = np.array([[0.5, 2.0], [0.25, 4.0], [3.0, 1.0], [7.0, 1.0]])
        y = oracle_mod.linear_f64(x, packed, s, 128)
        want0 = 0.5 * x[:, :128].sum(1) + 2.0 * x[:, 128:].sum(1)
        want1 = -(0.25 * x[:, :128].sum(1) + 4.0 * x[:, 128:].sum(1))
        np.testing.assert_allclose(y[:, 0], want0, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(y[:, 1], want1, rtol=1e-13, atol=1e-13)
    assert np.all(y[:, 2] == 0.0) and np.all(y[:, 3] == 0.0)
    assert y.shape == (M, N)


def test_one_hot_weight_picks_one_input(oracle_mod):
    rng = np.random.default_rng(3)
    M, K = 2, 512
    x = rng.standard_normal((M, K))
    for k in (0, 1, 2, 3, 127, 128, 300, 511):
        for code, sign in ((1, 1.0), (2, -1.0)):
            packed = np.zeros((1, K // 4), dtype=np.uint8)
            packed[0, k // 4] = code << (2 * (k % 4))
            s = np.full((1, K // 128), 0.0)
            s[0, k // 128] = 0.75
            y = oracle_mod.linear_f64(x, packed, s, 128)
            assert np.array_equal(y[:, 0], sign * 0.75 * x[:, k])
            y = oracle_mod.linear_f64(x, packed, np.array([1.5]), 0)
            assert np.array_equal(y[:, 0], sign * 1.5 * x[:, k])


@pytest.mark.parametrize("G", [128, 256])
def test_group_isolation(oracle_mod, G):
    rng = np.random.default_rng(5)
    M, K, N = 2, 512, 3
    x = rng.standard_normal((M, K))
    packed = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    t = second_formulation(packed)
    for g in range(K // G):
        s = np.zeros((N, K // G))
        s[:, g] = 1.0
        y = oracle_mod.linear_f64(x, packed, s, G)
        want = x[:, g * G:(g + 1) * G] @ t[:, g * G:(g + 1) * G].T.astype(np.float64)
        np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("group_size", [0, 128, 64, 256])
def test_matches_library_matmul(oracle_mod, group_size):
    """The oracle equals numpy's fp64 matmul of x and the dequantised weight
    (t * s broadcast per row / per group) to rounding."""
    rng = np.random.default_rng(11)
    M, N, K = 5, 33, 512
    x = rng.standard_normal((M, K))
    packed = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    t = second_formulation(packed).astype(np.float64)
    if group_size == 0:
        s = rng.uniform(0.01, 0.05, size=N)
        w = t * s[:, None]
    else:
        s = rng.uniform(0.01, 0.05, size=(N, K // group_size))
        w = t * np.repeat(s, group_size, axis=1)
    y = oracle_mod.linear_f64(x, packed, s, group_size)
    ref = np.matmul(x, w.T)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_linearity_and_row_independence(oracle_mod):
    rng = np.random.default_rng(13)
    M, N, K = 4, 9, 256
    x1 = rng.standard_normal((M, K))
    x2 = rng.standard_normal((M, K))
    packed = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    s = rng.uniform(0.01, 0.05, size=(N, 2))
    y1 = oracle_mod.linear_f64(x1, packed, s, 128)
    y2 = oracle_mod.linear_f64(x2, packed, s, 128)
    y12 = oracle_mod.linear_f64(2.0 * x1 - x2, packed, s, 128)
    np.testing.assert_allclose(y12, 2.0 * y1 - y2, rtol=1e-12, atol=1e-12)
    ys = oracle_mod.linear_f64(x1, packed, 4.0 * s, 128)
    assert np.array_equal(ys, 4.0 * y1)
    # a token row of the output depends only on that token row of x
    y_row = oracle_mod.linear_f64(x1[2:3], packed, s, 128)
    assert np.array_equal(y_row[0], y1[2])


def test_fused_rows_equal_shards(oracle_mod):
    """A fused layer (rows of several shards stacked, scale rows stacked at the
    same offsets) gives each shard's standalone result in its columns."""
    rng = np.random.default_rng(17)
    M, K = 3, 256
    shards = [5, 2, 2]
    x = rng.standard_normal((M, K))
    packs = [rng.integers(0, 256, size=(n, K // 4), dtype=np.uint8) for n in shards]
    scales = [rng.uniform(0.01, 0.05, size=(n, 2)) for n in shards]
    fused = oracle_mod.linear_f64(x, np.concatenate(packs), np.concatenate(scales), 128)
    off = 0
    for p, s in zip(packs, scales):
        part = oracle_mod.linear_f64(x, p, s, 128)
        assert np.array_equal(fused[:, off:off + p.shape[0]], part)
        off += p.shape[0]


# ---------------------------------------------------------------- SiLU-gated product
def _negate_codes(packed):
    """Swap codes 01 and 10 in every field: the same weights with the sign flipped."""
    b = packed.astype(np.uint16)
    out = np.zeros_like(b)
    for j in range(4):
        c = (b >> (2 * j)) & 3
        c = np.where(c == 1, 2, np.where(c == 2, 1, c))
        out |= c << (2 * j)
    return out.astype(np.uint8)


@pytest.mark.parametrize("group_size", [0, 128])
def test_silu_mul_odd_part_is_the_plain_product(oracle_mod, group_size):
    """silu(g) - silu(-g) = g for every g, so h(gate) - h(-gate) = g * u: pins the
    sign inside exp, which shard is the gate, and the rows' order."""
    rng = np.random.default_rng(23)
    M, N, K = 4, 7, 256
    x = rng.standard_normal((M, K))
    gate = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    up = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    ss = (2 * N,) if group_size == 0 else (2 * N, K // group_size)
    s = rng.uniform(0.2, 1.0, size=ss)
    h1 = oracle_mod.silu_mul_f64(x, np.concatenate([gate, up]), s, group_size)
    h2 = oracle_mod.silu_mul_f64(x, np.concatenate([_negate_codes(gate), up]), s, group_size)
    g = oracle_mod.linear_f64(x, gate, s[:N], group_size)
    u = oracle_mod.linear_f64(x, up, s[N:], group_size)
    np.testing.assert_allclose(h1 - h2, g * u, rtol=1e-12, atol=1e-12)


def test_silu_mul_point_values(oracle_mod):
    """One-hot weights give g = x_a, u = x_b: h = sigma(x_a) x_a x_b, checked at
    sigma(1) = 1 / (1 + 1/e) = 0.7310585786300049 and at g = 0 and g >> 0."""
    K = 64
    x = np.zeros((3, K))
    x[0, 0], x[0, 1] = 1.0, 2.0      # g = 1, u = 2
    x[1, 0], x[1, 1] = 0.0, 5.0      # g = 0: h = 0
    x[2, 0], x[2, 1] = 60.0, -0.5    # g = 60: silu(g) = g to 1e-24 relative
    t = np.zeros((2, K), dtype=np.int8)
    t[0, 0] = 1   # gate row reads x[:, 0]
    t[1, 1] = 1   # up row reads x[:, 1]
    packed, _ = oracle_mod.pack(t)
    h = oracle_mod.silu_mul_f64(x, packed, np.ones(2), 0)
    assert abs(h[0, 0] - 2.0 * 0.7310585786300049) < 1e-15
    assert h[1, 0] == 0.0
    assert abs(h[2, 0] - (-30.0)) < 1e-12


def test_silu_mul_zero_up_or_gate(oracle_mod):
    rng = np.random.default_rng(29)
    M, N, K = 2, 5, 128
    x = rng.standard_normal((M, K))
    gate = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    zero = np.zeros((N, K // 4), dtype=np.uint8)
    s = np.ones(2 * N)
    assert np.all(oracle_mod.silu_mul_f64(x, np.concatenate([gate, zero]), s, 0) == 0.0)
    assert np.all(oracle_mod.silu_mul_f64(x, np.concatenate([zero, gate]), s, 0) == 0.0)


def test_threads_do_not_change_results(oracle_mod):
    rng = np.random.default_rng(19)
    x = rng.standard_normal((3, 384))
    packed = rng.integers(0, 256, size=(50, 96), dtype=np.uint8)
    s = rng.uniform(0.01, 0.05, size=(50, 3))
    a = oracle_mod.linear_f64(x, packed, s, 128, nthreads=1)
    b = oracle_mod.linear_f64(x, packed, s, 128, nthreads=7)
    assert np.array_equal(a, b)


def test_bit_conversions_exact(oracle_mod):
    import torch
    v = torch.randn(1000, generator=torch.Generator().manual_seed(0))
    for dt, name in ((torch.float16, "f16"), (torch.bfloat16, "bf16")):
        t = v.to(dt)
        bits = t.view(torch.int16).numpy().view(np.uint16)
        got = oracle_mod.bits_to_f64(bits, name)
        assert np.array_equal(got, t.to(torch.float64).numpy())


# ------------------------------------------------------------------ zero-block map
# Blocks are 128 rows x 64 k.  Expected maps below are built from where the test
# itself put non-zero codes, by index arithmetic only (no decode).
def _expected_map(N, K, live_cells):
    RB, KB = (N + 127) // 128, (K + 63) // 64
    m = np.zeros((RB, (KB + 31) // 32), dtype=np.uint32)
    for rb, kb in live_cells:
        m[rb, kb // 32] |= np.uint32(1 << (kb % 32))
    return m


def test_block_mask_empty_and_reserved(oracle_mod):
    N, K = 300, 4160  # ragged in both: 3 row blocks, 65 k blocks
    for byte in (0x00, 0xFF, 0xF3, 0x3C):  # fields 00 / 11 only: every weight decodes to 0
        p = np.full((N, K // 4), byte, dtype=np.uint8)
        m, z = oracle_mod.block_mask(p)
        assert m.shape == (3, 3)
        assert not m.any() and z == 3 * 65


@pytest.mark.parametrize("code", [1, 2])
def test_block_mask_single_weight_positions(oracle_mod, code):
    """One +1 or -1 weight anywhere lights exactly its own block: rows 0, 127,
    128, 255, N-1 and k 0, 63, 64, 2047, K-1 (block edges, the ragged last blocks)."""
    N, K = 300, 4160
    for n in (0, 127, 128, 255, N - 1):
        for k in (0, 63, 64, 2047, K - 1):
            p = np.zeros((N, K // 4), dtype=np.uint8)
            p[n, k // 4] = code << (2 * (k % 4))
            m, z = oracle_mod.block_mask(p)
            assert np.array_equal(m, _expected_map(N, K, [(n // 128, k // 64)])), (n, k)
            assert z == 3 * 65 - 1


def test_block_mask_random_pattern(oracle_mod):
    """Live blocks carry random codes with at least one non-zero weight, zero blocks
    random 00 / 11 fields: the map is the pattern."""
    rng = np.random.default_rng(41)
    N, K = 520, 1920
    RB, KB = 5, 30
    live = rng.random((RB, KB)) < 0.7
    fields = rng.integers(0, 4, size=(N, K), dtype=np.uint8)
    for rb in range(RB):
        for kb in range(KB):
            r0, r1, k0, k1 = rb * 128, min(N, rb * 128 + 128), kb * 64, kb * 64 + 64
            blk = fields[r0:r1, k0:k1]
            if live[rb, kb]:
                blk[rng.integers(0, r1 - r0), rng.integers(0, 64)] = 1 + rng.integers(0, 2)
            else:
                blk[...] = 3 * (blk >= 2)  # 00 or 11
    packed = (fields[:, 0::4] | (fields[:, 1::4] << 2) | (fields[:, 2::4] << 4)
              | (fields[:, 3::4] << 6)).astype(np.uint8)
    m, z = oracle_mod.block_mask(packed)
    cells = [(rb, kb) for rb in range(RB) for kb in range(KB) if live[rb, kb]]
    assert np.array_equal(m, _expected_map(N, K, cells))
    assert z == int((~live).sum())
    # a second formulation: any non-zero in the unpacked block
    t, _ = oracle_mod.unpack(packed)
    for rb in range(RB):
        for kb in range(KB):
            assert bool(np.any(t[rb * 128:rb * 128 + 128, kb * 64:kb * 64 + 64])) == bool(live[rb, kb])


# ---------------------------------------------------------------- K % 4 != 0
def _tail_rows():
    for row in read_golden("tail_rows.txt"):
        K = int(row[0])
        packed = np.array([[int(b, 16) for b in row[1].split(",")]], dtype=np.uint8)
        t = np.array([[int(v) for v in row[2:]]], dtype=np.int8)
        assert t.shape[1] == K
        yield K, packed, t


def test_tail_rows_pack_and_unpack_by_hand(oracle_mod):
    for K, packed, t in _tail_rows():
        got, invalid = oracle_mod.pack(t)
        assert invalid == 0 and np.array_equal(got, packed), K
        back, reserved = oracle_mod.unpack(packed, K)
        assert reserved == 0 and np.array_equal(back, t), K


def test_tail_padding_fields_are_not_weights(oracle_mod):
    """Any codes in the padding fields (11 included) change neither the unpacked
    weights, nor the reserved count, nor the product, nor the zero-block map."""
    for K, packed, t in _tail_rows():
        pad = 4 * packed.shape[1] - K
        for fill in (1, 2, 3):
            dirty = packed.copy()
            for j in range(4 - pad, 4):
                dirty[0, -1] |= fill << (2 * j)
            back, reserved = oracle_mod.unpack(dirty, K)
            assert reserved == 0 and np.array_equal(back, t), (K, fill)
            x = 3.0 ** np.arange(K)[None, :]
            assert np.array_equal(oracle_mod.linear_f64(x, dirty, np.ones(1), 0),
                                  oracle_mod.linear_f64(x, packed, np.ones(1), 0))
        zero_row = np.zeros_like(packed)
        zero_row[0, -1] = 0xFF & ~((1 << (2 * (4 - pad))) - 1)  # padding fields all 11 / 01
        m, z = oracle_mod.block_mask(zero_row, K)
        assert not m.any() and z == 1


def test_tail_balanced_ternary_every_last_byte(oracle_mod):
    """K = 4q + r (r = 1, 2, 3): row n ends with byte n, x_k = 3^k, s = 1.  y[n]
    is the balanced-ternary number of the row's weights: the first r fields of
    byte n (from the golden table) times 3^(4q) -- the padding fields drop out."""
    table = table_from_golden()
    for K in (5, 6, 7, 9, 14):
        q, r = divmod(K, 4)
        packed = np.zeros((256, q + 1), dtype=np.uint8)
        packed[:, 0] = 0x49  # 1 -1 0 1
        packed[:, q] = np.arange(256, dtype=np.uint8)
        x = (3.0 ** np.arange(K))[None, :]
        y = oracle_mod.linear_f64(x, packed, np.ones(256), 0)[0]
        for b in range(256):
            head = 1 - 3 + 27
            tail = sum(table[(b >> (2 * j)) & 3] * 3 ** (4 * q + j) for j in range(r))
            assert y[b] == head + tail, (K, b)


def test_tail_per_channel_matches_library_matmul(oracle_mod):
    """Random K % 4 != 0 layers against numpy's matmul of the hand-decoded
    weights (second formulation of the table, padding fields random)."""
    rng = np.random.default_rng(23)
    for K in (1, 2, 3, 101, 333):
        N, M = 37, 5
        Kq = (K + 3) // 4
        packed = rng.integers(0, 256, size=(N, Kq), dtype=np.uint8)
        t = second_formulation(packed)[:, :K].astype(np.float64)
        x = rng.standard_normal((M, K))
        s = rng.uniform(0.01, 0.1, size=N)
        want = (x @ t.T) * s[None, :]
        np.testing.assert_allclose(oracle_mod.linear_f64(x, packed, s, 0), want,
                                   rtol=1e-12, atol=1e-12)
        got_t, _ = oracle_mod.unpack(packed, K)
        assert np.array_equal(got_t, t.astype(np.int8))
