"""GPU parity for rope_rows fused into the append: rotated q and k (and the
copied v) against the oracle's rope at the pages' precision, then decode
attention on the rotated inputs against the oracle.  Rotated values must
agree exactly except where a libm and a CUDA cos/sin/exp/log differ by an
ulp in a table entry (the library takes the inverse frequencies from the
host's libm, as the oracle does, and evaluates cos/sin in fp64, so such
differences are rare); a value may then move by one table ulp (bounded
below)."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_gb300 as pgd
from pgd_inputs import Workload, bf16_bits, layout_from_contexts, make_batch, make_rows_batch
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THETA = 1e6


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def as_float(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_rotated(got_bits, want_bits, src_bits, what):
    """Exact, or off by at most one bf16 table ulp on cos and sin (times the
    pair's inputs) plus one output ulp; at most 0.1 % of values may differ."""
    got, want = as_float(got_bits), as_float(want_bits)
    d = src_bits.shape[-1]
    src = as_float(src_bits)
    pair = np.abs(src[..., : d // 2]) + np.abs(src[..., d // 2:])
    pair = np.concatenate([pair, pair], axis=-1)
    bound = 2.0 ** -7 * pair + 2.0 ** -7 * np.abs(want)
    diff = np.abs(got - want)
    assert np.all(diff <= bound), f"{what}: max excess {np.max(diff - bound)}"
    frac = np.mean(got_bits != want_bits)
    assert frac <= 0.001, f"{what}: {frac:.4f} of values differ"


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (14, 2, 64), (64, 8, 64)])
def test_rope_append_then_decode(hq, hkv, d):
    wl = Workload("rope", rows=8, q_heads=hq, kv_heads=hkv, head_dim=d, ctx_lo=1,
                  ctx_hi=32768, sinks=hq == 64)
    contexts = [1, 2, 64, 65, 1000, 4097, 20000, 32768]
    lay = layout_from_contexts(wl, contexts, seed=40 + d)
    b = make_batch(wl, seed=41 + hq, device=DEV, layout=lay)
    q0, k0 = bf16_bits(b.q).copy(), bf16_bits(b.k_new).copy()
    k_pool_host, v_pool_host = bf16_bits(b.k_pool).copy(), bf16_bits(b.v_pool).copy()
    q = b.q.clone()
    pgd.rope_append_paged(q, b.k_new, b.v_new, b.table, b.positions, b.k_pool, b.v_pool,
                          theta=THETA)
    assert pgd.get_device_error() == pgd.OK
    want_q = oracle.rope(q0, lay.positions, THETA)
    want_k = oracle.rope(k0, lay.positions, THETA)
    check_rotated(bf16_bits(q), want_q, q0, "q")
    # the pool: rotated k and the copied v at each row's slot, nothing else touched
    slots = oracle.page_slots(lay.table, lay.positions, 64, lay.num_pages)
    geo = dict(kv_heads=hkv, head_dim=d, page_size=64, num_pages=lay.num_pages)
    oracle.write_tokens(k_pool_host, want_k, slots, **geo)
    oracle.write_tokens(v_pool_host, bf16_bits(b.v_new), slots, **geo)
    got_pool = bf16_bits(b.k_pool)
    tiles = got_pool.reshape(lay.num_pages, hkv, 64, d)
    want_tiles = k_pool_host.reshape(lay.num_pages, hkv, 64, d)
    for r, s in enumerate(slots):
        page, off = divmod(int(s), 64)
        check_rotated(tiles[page, :, off], want_tiles[page, :, off], k0[r], f"k row {r}")
        tiles[page, :, off] = want_tiles[page, :, off]      # compared; now mask it out
    assert np.array_equal(tiles.reshape(-1), k_pool_host)
    assert np.array_equal(bf16_bits(b.v_pool), v_pool_host)
    # attention on the rotated inputs: the oracle uses its own rotation throughout
    out = pgd.paged_decode_attention(q, b.k_pool, b.v_pool, b.table, b.positions, b.sinks,
                                     0, wl.scale, num_kv_heads=hkv)
    assert pgd.get_device_error() == pgd.OK
    want, _, _ = oracle.decode_paged(want_q, k_pool_host, v_pool_host, lay.table, lay.positions,
                                     kv_heads=hkv, num_pages=lay.num_pages,
                                     sinks=None if b.sinks is None else b.sinks.cpu().numpy(),
                                     scale=wl.scale)
    compare(out, want, f"rope+decode {hq}/{hkv} d{d}")


def test_rope_append_explicit_slots_and_inactive_rows():
    wl = Workload("rope_slots", rows=4, q_heads=8, kv_heads=2, head_dim=64, ctx_lo=1,
                  ctx_hi=300)
    lay = layout_from_contexts(wl, [10, 0, 200, 64], seed=42, num_pages=12)
    b = make_batch(wl, seed=43, device=DEV, layout=lay)
    slots = torch.tensor([5 * 64 + 9, 3 * 64, 11 * 64 + 7, 2 * 64 + 63], dtype=torch.int32,
                         device=DEV)
    q0 = b.q.clone()
    k_host = bf16_bits(b.k_pool).copy()
    pgd.rope_append_paged(b.q, b.k_new, b.v_new, None, b.positions, b.k_pool, b.v_pool,
                          theta=THETA, slots=slots)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(b.q[1], q0[1])                       # inactive row untouched
    want_k = oracle.rope(bf16_bits(b.k_new), lay.positions, THETA)
    tiles = bf16_bits(b.k_pool).reshape(12, 2, 64, 64)
    for r, s in enumerate(slots.tolist()):
        if lay.positions[r] < 0:
            continue
        page, off = divmod(s, 64)
        check_rotated(tiles[page, :, off], want_k[r], bf16_bits(b.k_new)[r], f"slot row {r}")
    # the inactive row's slot was not written
    assert np.array_equal(tiles[3, :, 0], k_host.reshape(12, 2, 64, 64)[3, :, 0])


def test_rope_append_dense_rows():
    wl = Workload("rope_rows", rows=3, q_heads=16, kv_heads=4, head_dim=128, ctx_lo=1,
                  ctx_hi=256)
    rb = make_rows_batch(wl, 44, DEV, contexts=[1, 130, 256])
    q0, k0 = bf16_bits(rb.q).copy(), bf16_bits(rb.k_new).copy()
    pgd.rope_append_paged(rb.q, rb.k_new, rb.v_new, None, rb.positions, rb.cache_k, rb.cache_v,
                          theta=THETA, layout=pgd.ROW_MAJOR, max_pages_per_row=rb.max_seq // 64)
    assert pgd.get_device_error() == pgd.OK
    check_rotated(bf16_bits(rb.q), oracle.rope(q0, rb.positions_np, THETA), q0, "q dense")
    want_k = oracle.rope(k0, rb.positions_np, THETA)
    cache = bf16_bits(rb.cache_k)
    for r, n in enumerate(rb.positions_np):
        check_rotated(cache[r, :, n], want_k[r], k0[r], f"dense row {r}")
        assert np.array_equal(bf16_bits(rb.cache_v)[r, :, n], bf16_bits(rb.v_new)[r])


def test_rope_append_bad_page_is_reported_and_row_left_alone():
    wl = Workload("rope_bad", rows=2, q_heads=4, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=128)
    lay = layout_from_contexts(wl, [5, 70], seed=45, num_pages=4)
    b = make_batch(wl, seed=46, device=DEV, layout=lay)
    table = b.table.clone()
    table[1, 1] = 99
    q0 = b.q.clone()
    pgd.rope_append_paged(b.q, b.k_new, b.v_new, table, b.positions, b.k_pool, b.v_pool,
                          theta=THETA)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.equal(b.q[1], q0[1]) and not torch.equal(b.q[0], q0[0])
