"""GPU parity of unip_rope_append_kv (through the C ABI) against the fp64
rotary-embedding oracle, and a chunked-prefill chain driven by the library's
step builder: rotary embedding + paged-cache append + attention, step after
step, against one-shot attention of every request's whole sequence.

Tolerance of the rotation (derived from the arithmetic): the kernel forms
each output in fp32 from bf16 inputs with an angle error below 3e-7 rad, so
before rounding it is within 1e-6 * max|input pair| of the exact value; bf16
rounding to nearest even adds at most 2^-8 of the magnitude.  Bits equal the
exact value rounded to bf16, except where it lies within that fp32 error of a
rounding midpoint; such elements are rare, and off by one unit in the last
place wherever the result is at least 2^-10 of its input pair (smaller
results come from cancellation and are held to the absolute bound)."""
import zlib

import numpy as np
import pytest

from oracle import rope as orope
from sparsified_long_context_gb300 import workloads as W

from gpu_harness import MAX_ABS, MEAN_ABS, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SENTINEL = 0x1234


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _round_bf16(x64):
    return W.f32_to_bf16_bits(x64.astype(np.float32))


def _check_rotation(got_bits, x_bits, positions, theta, interleaved, what):
    exact = orope.rope(orope.bf16_bits_to_f64(x_bits), positions, theta, interleaved)
    got = orope.bf16_bits_to_f64(got_bits)
    pair_mag = np.abs(orope.bf16_bits_to_f64(x_bits))
    d = x_bits.shape[-1]
    if interleaved:
        m = np.maximum(pair_mag[..., 0::2], pair_mag[..., 1::2]).repeat(2, axis=-1)
    else:
        m = np.tile(np.maximum(pair_mag[..., : d // 2], pair_mag[..., d // 2:]), 2)
    bound = 2.0 ** -8 * np.abs(exact) + 1e-6 * m + 1e-30
    err = np.abs(got - exact)
    assert np.all(err <= bound), f"{what}: worst err / bound {np.max(err / bound):.3f}"
    ref_bits = _round_bf16(exact)
    diff = got_bits != ref_bits
    assert diff.mean() <= 1e-3, f"{what}: {diff.mean():.2e} of elements not the rounded exact value"
    # Where the result is not much smaller than its inputs, the fp32 error is
    # below one bf16 unit, so rounding can only land on the neighbouring value.
    big = diff & (np.abs(exact) >= 2.0 ** -10 * m)
    step = np.abs(got_bits[big].astype(np.int32) - ref_bits[big].astype(np.int32))
    assert np.all(step == 1), f"{what}: differences larger than one unit in the last place"


CASES = [
    # name, lengths, H_q, H_kv, D, theta, interleaved, position kind
    ("packed_restarted", [37, 100, 64, 255], 4, 2, 64, 10000.0, False, "restart"),
    ("packed_restarted_inter", [37, 100, 64, 255], 4, 2, 64, 10000.0, True, "restart"),
    ("llama_shape_far_positions", [1001], 32, 8, 128, 500000.0, False, "random"),
    ("llama_shape_far_positions_inter", [1001], 32, 8, 128, 500000.0, True, "random"),
    ("chunk_continuation", [513], 16, 16, 128, 10000.0, False, "offset"),
    ("narrow_heads", [9], 2, 1, 16, 10000.0, False, "restart"),
    ("wide_heads", [40], 2, 2, 256, 1000000.0, True, "random"),
    ("negative_positions_inter", [300], 8, 2, 64, 10000.0, True, "signed"),
]


@pytest.mark.parametrize("name,lengths,hq,hkv,d,theta,inter,poskind", CASES, ids=[c[0] for c in CASES])
def test_rope_and_append_match_oracle(name, lengths, hq, hkv, d, theta, inter, poskind):
    from sparsified_long_context_gb300 import binding as B
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    n = sum(lengths)
    if poskind == "restart":
        positions = np.concatenate([np.arange(L) for L in lengths]).astype(np.int32)
    elif poskind == "offset":
        positions = (np.arange(n) + (1 << 20) + 12345).astype(np.int32)
    elif poskind == "signed":
        positions = rng.integers(-(1 << 21), 1 << 21, n).astype(np.int32)   # the rotation is defined for any integer
    else:
        positions = rng.integers(0, 1 << 22, n).astype(np.int32)
    q = W._normal_bf16(rng, (n, hq, d))
    k = W._normal_bf16(rng, (n, hkv, d))
    v = W._normal_bf16(rng, (n, hkv, d))
    page = 16
    num_pages = -(-n // page) + 3
    slots = rng.permutation(num_pages * page)[:n].astype(np.int32)
    slots[rng.random(n) < 0.1] = -1                                      # padding tokens: not appended
    B.unip_get_device_status(clear=True)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    kc = torch.full((num_pages, page, hkv, d), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    vc = torch.full((num_pages, page, hkv, d), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    pos_d = torch.from_numpy(positions).cuda()
    slot_d = torch.from_numpy(slots).cuda()
    B.unip_rope_append_kv(qd, kd, vd, pos_d, num_heads_q=hq, num_heads_kv=hkv, head_dim=d, rope_theta=theta,
                          interleaved=inter, slot_mapping=slot_d, k_cache=kc, v_cache=vc, page_size=page)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    q_got, k_got = _bits(qd), _bits(kd)
    _check_rotation(q_got, q, positions, theta, inter, f"{name} q")
    _check_rotation(k_got, k, positions, theta, inter, f"{name} k")
    assert np.array_equal(_bits(vd), v)                                   # v is not modified
    kcb = _bits(kc).reshape(num_pages * page, hkv, d)
    vcb = _bits(vc).reshape(num_pages * page, hkv, d)
    live = slots >= 0
    assert np.array_equal(kcb[slots[live]], k_got[live])                  # the rotated k, bit for bit
    assert np.array_equal(vcb[slots[live]], v[live])
    untouched = np.ones(num_pages * page, bool)
    untouched[slots[live]] = False
    assert np.all(kcb[untouched] == SENTINEL) and np.all(vcb[untouched] == SENTINEL)


def test_append_only_leaves_q_and_k_alone():
    from sparsified_long_context_gb300 import binding as B
    rng = np.random.default_rng(11)
    n, hq, hkv, d, page = 70, 4, 2, 128, 16
    q, k, v = (W._normal_bf16(rng, (n, h, d)) for h in (hq, hkv, hkv))
    slots = rng.permutation(5 * page)[:n].astype(np.int32)
    qd, kd, vd = _dev(q), _dev(k), _dev(v)
    kc = torch.zeros((5, page, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    B.unip_rope_append_kv(qd, kd, vd, None, num_heads_q=hq, num_heads_kv=hkv, head_dim=d, rope_theta=0.0,
                          slot_mapping=torch.from_numpy(slots).cuda(), k_cache=kc, v_cache=vc, page_size=page)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(qd), q) and np.array_equal(_bits(kd), k)
    assert np.array_equal(_bits(kc).reshape(-1, hkv, d)[slots], k)
    assert np.array_equal(_bits(vc).reshape(-1, hkv, d)[slots], v)


def test_slot_beyond_the_cache_is_reported_and_skipped():
    from sparsified_long_context_gb300 import binding as B
    rng = np.random.default_rng(12)
    n, hq, hkv, d, page, num_pages = 20, 2, 2, 64, 16, 2
    q, k, v = (W._normal_bf16(rng, (n, h, d)) for h in (hq, hkv, hkv))
    slots = np.arange(n, dtype=np.int32)
    slots[5] = num_pages * page + 7                                       # out of range: must not be written
    B.unip_get_device_status(clear=True)
    kc = torch.full((num_pages, page, hkv, d), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    vc = torch.full_like(kc, 0)
    kd = _dev(k)
    B.unip_rope_append_kv(_dev(q), kd, _dev(v), torch.arange(n, dtype=torch.int32, device="cuda"), num_heads_q=hq,
                          num_heads_kv=hkv, head_dim=d, slot_mapping=torch.from_numpy(slots).cuda(), k_cache=kc,
                          v_cache=vc, page_size=page)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st & 0x40, B.describe_status(st)
    kcb = _bits(kc).reshape(-1, hkv, d)
    ok = np.arange(n) != 5
    assert np.array_equal(kcb[slots[ok]], _bits(kd)[ok])
    assert np.all(kcb[5] == SENTINEL)                                     # slot 5 belongs to no token now


def test_chunked_steps_with_rope_match_one_shot():
    """Requests go through the step builder's mixed steps (decodes first, then
    64-aligned prompt chunks under a 256-token budget).  Each step rotates its
    tokens' q and k by their absolute positions, appends k and v to the paged
    cache at the step's slots and runs attention over the cached prefix plus
    the step's own tokens.  Every token's output equals one-shot causal
    attention over its request's whole (rotated) sequence."""
    from sparsified_long_context_gb300 import binding as B
    rng = np.random.default_rng(21)
    hq, hkv, d, page, theta = 8, 2, 128, 16, 10000.0
    reqs = [(300, 4), (77, 3), (513, 2), (1, 5), (190, 1)]
    seqs = []
    for (L, m) in reqs:
        T = L + m - 1
        seqs.append(tuple(W._normal_bf16(rng, (T, h, d)) for h in (hq, hkv, hkv)))
    num_pages, max_pages = 160, 64
    sb = B.StepBuilder(256, page, num_pages, max_pages, 16, 64)
    for (L, m) in reqs:
        sb.add(L, m)
    kc = torch.zeros((num_pages, page, hkv, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    outs = [np.full((s[0].shape[0], hq, d), np.nan) for s in seqs]
    B.unip_get_device_status(clear=True)
    steps = 0
    while True:
        st = sb.next()
        cu = st["cu_seqlens"]
        if len(cu) == 1:
            break
        steps += 1
        rid, pos = st["request_ids"], st["positions"]
        owner = np.repeat(rid, np.diff(cu))
        q = np.stack([seqs[r][0][p] for r, p in zip(owner, pos)])
        k = np.stack([seqs[r][1][p] for r, p in zip(owner, pos)])
        v = np.stack([seqs[r][2][p] for r, p in zip(owner, pos)])
        qd, kd, vd = _dev(q), _dev(k), _dev(v)
        pos_d = torch.from_numpy(pos).cuda()
        B.unip_rope_append_kv(qd, kd, vd, pos_d, num_heads_q=hq, num_heads_kv=hkv, head_dim=d, rope_theta=theta,
                              slot_mapping=torch.from_numpy(st["slot_mapping"]).cuda(), k_cache=kc, v_cache=vc,
                              page_size=page)
        out = torch.empty_like(qd)
        B.unip_prefill_attention(qd, kd, vd, torch.from_numpy(cu).cuda(), pos_d, out, None, num_heads_q=hq,
                                 num_heads_kv=hkv, head_dim=d, k_cache=kc, v_cache=vc,
                                 block_table=torch.from_numpy(st["block_table"]).cuda(), page_size=page)
        o = out.float().cpu().numpy().astype(np.float64)
        for i, (r, p) in enumerate(zip(owner, pos)):
            outs[r][p] = o[i]
    torch.cuda.synchronize()
    s = B.unip_get_device_status(clear=True)
    assert s == 0, B.describe_status(s)
    assert steps >= 6
    import oracle
    for r, (qb, kb, vb) in enumerate(seqs):
        T = qb.shape[0]
        pos = np.arange(T)
        q_r = _round_bf16(orope.rope(orope.bf16_bits_to_f64(qb), pos, theta))
        k_r = _round_bf16(orope.rope(orope.bf16_bits_to_f64(kb), pos, theta))
        ref, _ = oracle.attention(q_r, k_r, vb, np.array([0, T], np.int32), pos.astype(np.int32), hq, hkv, d)
        assert_close(outs[r], ref, MAX_ABS, MEAN_ABS, what=f"request {r}")
