"""The step before decode on the GPU (QKV norm + RoPE + paged-cache write)
against the fp64 oracle, through the C ABI.

Tolerance (derived from the arithmetic): the kernel normalises and rotates in
fp32 from the exact bf16 inputs and rounds once to bf16, so an element may be
off by half a bf16 ulp of its value (2^-9 relative) plus fp32 rounding of the
norm, the table entries and the rotation, a few 2^-24 of the row's largest
element. The test allows |gpu - oracle| <= 2^-8 |oracle| + 2^-16 max|row|.
The RoPE table is fp64 rounded to fp32: within 2^-24 of the oracle's value
(plus the fp64 angle difference, below 1e-10 at 131072 positions).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import binding as b
from paged_gqa_decode_global_gb300 import inputs as synth

pytestmark = pytest.mark.gpu


def _dev(t):
    return None if t is None else t.cuda()


def _desc(li):
    return b.layer_desc(li.num_q_heads, li.num_kv_heads, li.head_dim, li.page_size, li.num_pages,
                        li.block_tables.shape[1], li.window, li.v_pool is None)


def _oracle(pi):
    li = pi.layer
    return oracle.prepare_qkv(synth.bits_u16(pi.q_in), synth.bits_u16(pi.k_in),
                              None if pi.v_in is None else synth.bits_u16(pi.v_in), synth.bits_u16(pi.q_w),
                              synth.bits_u16(pi.k_w), None if pi.v_w is None else synth.bits_u16(pi.v_w),
                              li.block_tables.cpu().numpy(), li.seq_lens.cpu().numpy(), li.num_pages,
                              li.page_size, pi.rot, pi.theta, pi.eps)


def _close(got_bf16, exp_f64, what):
    got = got_bf16.float().cpu().double().numpy()
    exp = np.asarray(exp_f64)
    bound = 2.0 ** -8 * np.abs(exp) + 2.0 ** -16 * np.abs(exp).max(axis=-1, keepdims=True)
    err = np.abs(got - exp)
    assert (err <= bound).all(), f"{what}: worst excess {(err - bound).max():.3g}"


class GpuPrepare:
    """Device copies of a PrepareInputs and one call of the fused op."""

    def __init__(self, pi):
        self.pi = pi
        li = pi.layer
        self.q_in, self.k_in, self.v_in = _dev(pi.q_in), _dev(pi.k_in), _dev(pi.v_in)
        self.q_w, self.k_w, self.v_w = _dev(pi.q_w), _dev(pi.k_w), _dev(pi.v_w)
        self.table = _dev(li.block_tables)
        self.seq = _dev(li.seq_lens)
        self.k_pool = _dev(li.k_pool).clone()
        self.v_pool = None if li.v_pool is None else _dev(li.v_pool).clone()
        self.q_out = torch.full_like(self.q_in, 7.0)  # sentinel: rows not written keep it
        self.flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.cos_sin = None
        if pi.rot > 0:
            self.cos_sin = torch.empty(pi.max_positions, pi.rot, dtype=torch.float32, device="cuda")
            b.paged_decode_rope_table(pi.theta, pi.rot, pi.max_positions, self.cos_sin)

    def launch(self, seq=None, table=None, stream=None):
        pi, li = self.pi, self.pi.layer
        b.paged_decode_qkv_norm_rope_write(_desc(li), pi.rot, pi.max_positions, pi.eps, self.q_in, self.k_in,
                                           self.v_in, self.q_w, self.k_w, self.v_w, self.cos_sin,
                                           self.table if table is None else table,
                                           self.seq if seq is None else seq, self.q_out, self.k_pool,
                                           self.v_pool, self.flags, stream)

    def run(self, seq=None, table=None):
        self.launch(seq, table)
        torch.cuda.synchronize()
        return int(self.flags.item())


LAYERS = [
    # name, lens, Hq, Hkv, d, window, kv_shared, P, rot, theta
    ("global d512 K!=V", [1, 16, 17, 1000, 65537], 16, 4, 512, 0, False, 16, 128, 1e6),
    ("global d512 K=V", [2, 33, 4096], 16, 4, 512, 0, True, 16, 128, 1e6),
    ("sliding d256", [4100, 4200, 1, 15], 16, 8, 256, 1024, False, 16, 256, 1e4),
    ("sliding d256 K=V, P32", [31, 32, 65, 7], 8, 8, 256, 1024, True, 32, 64, 1e4),
    ("d512 no rotation", [5, 77], 8, 2, 512, 0, False, 16, 0, 1e4),
]


def _make(name, lens, Hq, Hkv, d, window, kvs, P, rot, theta, seed=11):
    pool = sum((L + P - 1) // P for L in lens) + 3
    li = synth.make_layer(name, lens, Hq, Hkv, d, window=window, kv_shared=kvs, pool_pages=pool, page_size=P,
                          seed=seed)
    return synth.make_prepare(li, rot=rot, theta=theta, seed=seed)


@pytest.mark.parametrize("rot,theta,n_pos", [(64, 1e6, 131072), (256, 1e4, 5000), (2, 100.0, 7)])
def test_rope_table_matches_oracle(rot, theta, n_pos):
    t = torch.empty(n_pos, rot, dtype=torch.float32, device="cuda")
    b.paged_decode_rope_table(theta, rot, n_pos, t)
    torch.cuda.synchronize()
    exp = oracle.rope_table(rot, theta, n_pos)
    got = t.cpu().double().numpy()
    assert np.abs(got - exp).max() <= 2.0 ** -24 + 1e-10


def _random_layers(n=30, seed=20261206):
    """Seeded random shapes of the step before decode: head_dim, groups 1..16,
    K=V, page sizes of 16..64 tokens, rotary dims from none to the whole head,
    windows, ragged lengths."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([256, 512]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 3, 4, 8, 16]))
        kvs = bool(rng.random() < 0.4)
        P = int(rng.choice([16, 32, 48, 64]))
        rot = int(rng.choice([0, 2, 64, d // 4, d // 2, d]))
        theta = float(rng.choice([100.0, 1e4, 1e6]))
        window = int(rng.choice([0, 1024]))
        B = int(rng.integers(1, 7))
        lens = [max(1, int(x)) for x in np.exp(rng.uniform(0.0, np.log(5000), B))]
        if B * max(lens) * Hkv * d > 40_000_000:  # keeps the host-side pools small
            continue
        name = f"rnd{len(out)} d{d} G{G} Hkv{Hkv} kvs{int(kvs)} P{P} rot{rot} W{window}"
        out.append((name, lens, G * Hkv, Hkv, d, window, kvs, P, rot, theta))
    return out


RANDOM_LAYERS = _random_layers()


@pytest.mark.parametrize("case", LAYERS, ids=[c[0] for c in LAYERS])
def test_prepare_matches_oracle(case):
    _check_prepare(case)


@pytest.mark.parametrize("case", RANDOM_LAYERS, ids=[c[0] for c in RANDOM_LAYERS])
def test_prepare_random_shapes_match_oracle(case):
    _check_prepare(case)


def _check_prepare(case):
    pi = _make(*case)
    li = pi.layer
    g = GpuPrepare(pi)
    k_before = g.k_pool.clone()
    v_before = None if g.v_pool is None else g.v_pool.clone()
    assert g.run() == 0
    q, k, v, page, row = _oracle(pi)
    _close(g.q_out, q, "q_out")
    written = torch.zeros(li.num_pages, li.page_size, dtype=torch.bool, device="cuda")
    for bi in range(li.batch):
        _close(g.k_pool[page[bi], :, row[bi], :], k[bi], f"k row of request {bi}")
        if g.v_pool is not None:
            _close(g.v_pool[page[bi], :, row[bi], :], v[bi], f"v row of request {bi}")
        written[page[bi], row[bi]] = True
    # every other row of the pools is untouched, bit for bit
    keep = (~written)[:, None, :, None].expand_as(g.k_pool)
    assert torch.equal(g.k_pool[keep], k_before[keep])
    if g.v_pool is not None:
        assert torch.equal(g.v_pool[keep], v_before[keep])


def test_unit_v_weight_and_repeat_determinism():
    pi = _make("d256 unit v weight", [9, 300], 8, 4, 256, 0, False, 16, 256, 1e4)
    pi.v_w = None
    g = GpuPrepare(pi)
    assert g.run() == 0
    q, k, v, page, row = _oracle(pi)
    for bi in range(pi.layer.batch):
        _close(g.v_pool[page[bi], :, row[bi], :], v[bi], "v row, unit weight")
    first = (g.q_out.clone(), g.k_pool.clone(), g.v_pool.clone())
    assert g.run() == 0
    assert torch.equal(first[0], g.q_out) and torch.equal(first[1], g.k_pool) and torch.equal(first[2], g.v_pool)


def _prepared_decode_oracle(pi):
    """The oracle's step, its rows rounded to bf16 into a host copy of the
    pools, then its decode."""
    li = pi.layer
    q, k, v, page, row = _oracle(pi)
    kpool = li.k_pool.clone()
    vpool = None if li.v_pool is None else li.v_pool.clone()
    for bi in range(li.batch):
        kpool[page[bi], :, row[bi], :] = torch.from_numpy(k[bi]).to(torch.bfloat16)
        if vpool is not None:
            vpool[page[bi], :, row[bi], :] = torch.from_numpy(v[bi]).to(torch.bfloat16)
    q16 = torch.from_numpy(q).to(torch.bfloat16)
    return oracle.decode(synth.bits_u16(q16), synth.bits_u16(kpool), None if vpool is None else synth.bits_u16(vpool),
                         li.block_tables.numpy(), li.seq_lens.numpy(), li.scale, li.window)


def _decode_after(g, early_kv, stream=None):
    """Stage 1 (+ merge) on the prepared cache, launched behind whatever is
    on the stream; plan.early_kv as given."""
    li = g.pi.layer
    plan = b.paged_decode_plan(_desc(li), li.seq_lens.tolist(), torch.cuda.get_device_properties(0).multi_processor_count)
    plan.early_kv = early_kv
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g.q_out)
    if li.window > 0:
        b.paged_decode_window(plan, g.q_out, g.k_pool, g.v_pool, g.table, g.seq, li.window, li.scale, ws, out, stream)
    else:
        b.paged_decode_global(plan, g.q_out, g.k_pool, g.v_pool, g.table, g.seq, li.scale, ws, out, stream)
    b.paged_decode_merge(plan, ws, out, stream)
    return out, plan, ws


def _check_decode(out, exp):
    got = out.float().cpu().double().numpy()
    assert np.abs(got - exp).max() <= 2e-2
    cos = (got * exp).sum() / np.sqrt((got * got).sum() * (exp * exp).sum())
    assert cos > 0.9995


@pytest.mark.parametrize("case", [LAYERS[0], LAYERS[2], LAYERS[1]], ids=["global", "sliding", "global K=V"])
def test_prepare_then_decode_matches_oracle(case):
    """GPU: fused step, a host sync, then decode; against the oracle's step + decode."""
    pi = _make(*case, seed=23)
    g = GpuPrepare(pi)
    assert g.run() == 0
    out, _, _ = _decode_after(g, 0)
    torch.cuda.synchronize()
    _check_decode(out, _prepared_decode_oracle(pi))


@pytest.mark.parametrize("case", [LAYERS[0], LAYERS[2], LAYERS[1], LAYERS[3]],
                         ids=["global", "sliding", "global K=V", "sliding K=V P32"])
def test_prepare_then_early_decode_matches_oracle(case):
    """The fused step and an early_kv decode back to back on one stream, no
    host sync between: stage 1 may copy older rows while the step runs, but
    must read each request's new row (and q) only after it. The new rows hold
    a large sentinel before the step, so a copy taken too early shows in the
    output; short requests put the new row in the first pipeline stages."""
    pi = _make(*case, seed=29)
    li = pi.layer
    g = GpuPrepare(pi)
    P = li.page_size
    for bi, L in enumerate(li.seq_lens.tolist()):
        page = int(li.block_tables[bi, (L - 1) // P])
        g.k_pool[page, :, (L - 1) % P, :] = 64.0
        if g.v_pool is not None:
            g.v_pool[page, :, (L - 1) % P, :] = -64.0
    g.q_out.fill_(0.5)
    exp = _prepared_decode_oracle(pi)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.launch(stream=s)
        out, plan, ws = _decode_after(g, 1, stream=s)
    s.synchronize()
    assert int(g.flags.item()) == 0
    assert b.paged_decode_check_device_error(plan, ws, s) == 0
    _check_decode(out, exp)


def test_bad_length_and_bad_page_flags():
    pi = _make("flags", [20, 40, 60], 8, 2, 256, 0, False, 16, 256, 1e4)
    li = pi.layer
    g = GpuPrepare(pi)
    k_before = g.k_pool.clone()
    # request 0: length 0 (nothing written), request 1: beyond the table
    cap = li.block_tables.shape[1] * li.page_size
    seq = torch.tensor([0, cap + 1, 60], dtype=torch.int32, device="cuda")
    flags = g.run(seq=seq)
    assert flags == b.PD_DEVFLAG_BAD_SEQLEN
    assert (g.q_out[:2].float() == 7.0).all()  # untouched
    assert not (g.q_out[2].float() == 7.0).all()
    # request 2's page id outside the pool: q written, cache untouched
    g.flags.zero_()
    g.k_pool.copy_(k_before)
    g.q_out.fill_(7.0)
    table = g.table.clone()
    table[2, (60 - 1) // li.page_size] = li.num_pages + 5
    flags = g.run(table=table)
    assert flags == b.PD_DEVFLAG_BAD_PAGE
    assert not (g.q_out[2].float() == 7.0).all()
    q, k, v, page, row = _oracle(pi)
    for bi in (0, 1):
        _close(g.k_pool[page[bi], :, row[bi], :], k[bi], "k row")
    assert torch.equal(g.k_pool[page[2], :, row[2], :], k_before[page[2], :, row[2], :])


def test_position_beyond_rope_table_is_flagged():
    pi = _make("table", [10, 50], 8, 2, 256, 0, False, 16, 256, 1e4)
    pi.max_positions = 40  # position 49 has no row
    g = GpuPrepare(pi)
    assert g.run() == b.PD_DEVFLAG_BAD_SEQLEN
    assert (g.q_out[1].float() == 7.0).all()
    assert not (g.q_out[0].float() == 7.0).all()


def test_host_rejections():
    pi = _make("rej", [10], 8, 2, 256, 0, False, 16, 256, 1e4)
    li = pi.layer
    g = GpuPrepare(pi)
    fp8 = _desc(li)
    fp8.kv_dtype = b.PD_KV_FP8_E4M3
    lib = b.load_library()
    args = lambda desc, rot=pi.rot: (desc, rot, pi.max_positions, pi.eps, g.q_in, g.k_in, g.v_in, g.q_w, g.k_w, g.v_w,
                                     g.cos_sin, g.table, g.seq, g.q_out, g.k_pool, g.v_pool, g.flags)
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_qkv_norm_rope_write(*args(fp8))
    assert e.value.status == b.PD_ERR_UNSUPPORTED
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_qkv_norm_rope_write(*args(_desc(li), rot=3))
    assert e.value.status == b.PD_ERR_INVALID_ARG
    # a misaligned q_in
    q_mis = torch.empty(g.q_in.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + g.q_in.numel()]
    with pytest.raises(b.PagedDecodeError) as e:
        b.paged_decode_qkv_norm_rope_write(_desc(li), pi.rot, pi.max_positions, pi.eps, q_mis.view_as(g.q_in),
                                           g.k_in, g.v_in, g.q_w, g.k_w, g.v_w, g.cos_sin, g.table, g.seq,
                                           g.q_out, g.k_pool, g.v_pool, g.flags)
    assert e.value.status == b.PD_ERR_INVALID_ARG
    assert lib.paged_decode_rope_table(0.0, 64, 10, g.cos_sin.data_ptr(), None) == b.PD_ERR_INVALID_ARG
