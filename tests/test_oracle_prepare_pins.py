"""Pins the oracle of the step before decode (per-head RMS norm of q / k / v,
RoPE of q and k at the new token's position, the cache slot of its k / v rows)
to things other than itself (CPU only):

* hand-derived values: rows whose mean square is a perfect square, an eps that
  makes the norm exactly 1/2, a RoPE base whose second frequency is exactly
  1/10 (tests/golden/prepare_hand_examples.json, derivations in the file);
* the rotation written as multiplication by exp(i * angle) of complex numbers
  (numpy complex128), on random rows, partial and full rotary widths;
* invariants: the rotated q . k depends only on the distance of the two
  positions; a normalised row has mean square 1 and points along its input;
* the slot: writing the returned k / v rows there and decoding with a window
  of one token (the decode oracle, itself pinned) returns exactly that v row.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_global_gb300 import inputs as synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(x):
    return synth.bits_u16(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def _one(q, k, v, qw, kw, vw, L, rot, theta, eps, P=4):
    """One request, one q head, one KV head, d = len(q)."""
    d = len(q)
    pages = (L + P - 1) // P
    table = np.arange(pages, dtype=np.int32)[None, :]
    return oracle.prepare_qkv(_bits([[q]]), _bits([[k]]), None if v is None else _bits([[v]]), _bits(qw),
                              _bits(kw), None if vw is None else _bits(vw), table, np.array([L], np.int32),
                              num_pages=pages, page_size=P, rot=rot, theta=theta, eps=eps)


def test_hand_examples():
    with open(os.path.join(HERE, "golden", "prepare_hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        qo, ko, vo, page, row = _one(c["q"], c["k"], c.get("v"), c["q_w"], c["k_w"], c.get("v_w"), c["L"],
                                     c["rot"], c["theta"], c["eps"])
        for name, got in (("q", qo[0, 0]), ("k", ko[0, 0])) + ((("v", vo[0, 0]),) if vo is not None else ()):
            exp = np.array([eval(e, {"math": math}) if isinstance(e, str) else e for e in c["expect_" + name]])
            np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12, err_msg=f"{c['name']}: {name}")
        assert (int(page[0]), int(row[0])) == tuple(c["slot"]), c["name"]


def _random_case(B, Hq, Hkv, d, lens, rot, theta, kv_shared=False, seed=0, P=16):
    pool = sum((L + P - 1) // P for L in lens) + 2
    li = synth.make_layer("p", lens, Hq, Hkv, d, kv_shared=kv_shared, pool_pages=pool, page_size=P, seed=seed)
    pi = synth.make_prepare(li, rot=rot, theta=theta, seed=seed)
    return li, pi


def _run(pi, rot=None, v_w="given", lens=None):
    li = pi.layer
    seq = li.seq_lens.numpy() if lens is None else np.asarray(lens, np.int32)
    return oracle.prepare_qkv(synth.bits_u16(pi.q_in), synth.bits_u16(pi.k_in),
                              None if pi.v_in is None else synth.bits_u16(pi.v_in), synth.bits_u16(pi.q_w),
                              synth.bits_u16(pi.k_w),
                              None if (pi.v_w is None or v_w is None) else synth.bits_u16(pi.v_w),
                              li.block_tables.numpy(), seq, li.num_pages, li.page_size,
                              pi.rot if rot is None else rot, pi.theta, pi.eps)


def _complex_rotate(y, pos, rot, theta):
    half = rot // 2
    z = y[..., :half] + 1j * y[..., half:rot]
    freq = theta ** (-2.0 * np.arange(half) / rot)
    z = z * np.exp(1j * pos * freq)
    out = y.copy()
    out[..., :half] = z.real
    out[..., half:rot] = z.imag
    return out


@pytest.mark.parametrize("d,rot,theta,lens", [(8, 8, 100.0, [1, 2, 9]), (8, 2, 1e4, [5, 33]),
                                              (256, 256, 1e4, [4100, 17]), (512, 128, 1e6, [131072, 1000]),
                                              (256, 64, 1e6, [77, 65536])])
def test_rotation_equals_complex_multiplication(d, rot, theta, lens):
    li, pi = _random_case(len(lens), 4, 2, d, lens, rot, theta)
    q0, k0, v0, _, _ = _run(pi, rot=0)
    q1, k1, v1, _, _ = _run(pi)
    pos = (np.asarray(lens) - 1)[:, None, None]
    # the two sides round pos * theta^(-2i/rot) independently: an angle of
    # size A is known to about A * 2^-52, which bounds the difference
    atol = 1e-12 + 4 * float(pos.max()) * 2.0 ** -52 * max(np.abs(q0).max(), np.abs(k0).max())
    np.testing.assert_allclose(q1, _complex_rotate(q0, pos, rot, theta), rtol=0, atol=atol)
    np.testing.assert_allclose(k1, _complex_rotate(k0, pos, rot, theta), rtol=0, atol=atol)
    np.testing.assert_array_equal(v1, v0)  # v is never rotated


def test_rotated_dot_depends_only_on_distance():
    d, rot, theta = 64, 64, 1e4
    li, pi = _random_case(1, 2, 2, d, [300], rot, theta)
    dots = []
    for m, n in ((10, 3), (110, 103), (290, 283)):
        qm = _run(pi, lens=[m + 1])[0][0, 0]
        kn = _run(pi, lens=[n + 1])[1][0, 0]
        dots.append(float(qm @ kn))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-11)
    # and a different distance gives a different product
    qm = _run(pi, lens=[11])[0][0, 0]
    kn = _run(pi, lens=[6])[1][0, 0]
    assert abs(float(qm @ kn) - dots[0]) > 1e-6


def test_normalised_rows_have_unit_mean_square():
    d = 256
    li = synth.make_layer("p", [40, 3], 4, 2, d, pool_pages=8, seed=3)
    pi = synth.make_prepare(li, rot=0, seed=3)
    ones = torch.ones(d, dtype=torch.bfloat16)
    pi.q_w = pi.k_w = pi.v_w = ones
    pi.eps = 0.0
    q, k, v, _, _ = _run(pi)
    for y, x in ((q, pi.q_in), (k, pi.k_in), (v, pi.v_in)):
        np.testing.assert_allclose(np.mean(y ** 2, axis=-1), 1.0, rtol=1e-13)
        xd = x.to(torch.float64).numpy()
        c = y / xd
        np.testing.assert_allclose(c, np.broadcast_to(c[..., :1], c.shape), rtol=1e-13)
        assert (c > 0).all()
    # no v weight means unit weight
    _, _, v_none, _, _ = _run(pi, v_w=None)
    np.testing.assert_array_equal(v_none, v)


def test_pass_through_dims_beyond_rot():
    li, pi = _random_case(2, 4, 2, 256, [50, 700], 64, 1e6)
    q0, k0, _, _, _ = _run(pi, rot=0)
    q1, k1, _, _, _ = _run(pi)
    np.testing.assert_array_equal(q1[..., 64:], q0[..., 64:])
    np.testing.assert_array_equal(k1[..., 64:], k0[..., 64:])
    assert not np.allclose(q1[..., :64], q0[..., :64])


@pytest.mark.parametrize("kv_shared,P,lens", [(False, 16, [1, 16, 17, 100]), (True, 16, [33, 2]),
                                              (False, 32, [31, 32, 65])])
def test_slot_holds_the_newest_position(kv_shared, P, lens):
    """Rows written to the returned slot are exactly what a one-token window decodes."""
    li, pi = _random_case(len(lens), 4, 2, 8, lens, 8, 100.0, kv_shared=kv_shared, P=P)
    q, k, v, page, row = _run(pi)
    assert (page >= 0).all()
    zero = torch.zeros_like(li.k_pool)
    kpool, vpool = zero.clone(), None if kv_shared else zero.clone()
    for b in range(len(lens)):
        kpool[page[b], :, row[b], :] = torch.from_numpy(k[b]).to(torch.bfloat16)
        if not kv_shared:
            vpool[page[b], :, row[b], :] = torch.from_numpy(v[b]).to(torch.bfloat16)
    out = oracle.decode(synth.bits_u16(li.q), synth.bits_u16(kpool),
                        None if kv_shared else synth.bits_u16(vpool), li.block_tables.numpy(),
                        li.seq_lens.numpy(), li.scale, window=1)
    newest = torch.from_numpy(k if kv_shared else v).to(torch.bfloat16).to(torch.float64).numpy()
    G = li.num_q_heads // li.num_kv_heads
    np.testing.assert_array_equal(out, np.repeat(newest, G, axis=1))


def test_rope_table_matches_closed_form():
    t = oracle.rope_table(4, 100.0, 3)
    exp = np.array([[1, 1, 0, 0],
                    [math.cos(1), math.cos(0.1), math.sin(1), math.sin(0.1)],
                    [math.cos(2), math.cos(0.2), math.sin(2), math.sin(0.2)]])
    np.testing.assert_allclose(t, exp, rtol=0, atol=1e-15)


def test_bad_length_is_refused():
    li, pi = _random_case(1, 2, 1, 8, [5], 8, 100.0)
    with pytest.raises(oracle.OracleError):
        _run(pi, lens=[0])
    with pytest.raises(oracle.OracleError):
        _run(pi, lens=[li.block_tables.shape[1] * li.page_size + 1])
