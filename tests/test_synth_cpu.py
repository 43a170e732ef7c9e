"""The seeded input generators against their stated recipe (no GPU).

The parity tests and the bench both draw from weight_only_quantized_qgemv_gb300.synth;
these tests pin what they rely on: the seeds and laws of every workload, that
draws are reproducible and streams independent, that a compact store of some
experts holds exactly those experts' matrices (the full-size expert tests
compare the device's full store against it), that the ue8m0 expert workload
holds the same values as the f32 one, and the algorithmic bytes per call that
the bench's roofline divides by.
"""
import numpy as np
import pytest

from weight_only_quantized_qgemv_gb300 import synth


def test_seeds_follow_the_recipe():
    """seed = 1000 + workload index; the s = 4 case shares the s = 1 matrix with its own x stream."""
    seeds = {n: synth.workload(n).seed for n in synth.WORKLOADS}
    assert seeds == {"int8_row_1024x1024_s1": 1001, "int4_g32_16384x6144_s1": 1002,
                     "int4_g32_16384x6144_s4": 1002, "int3_g64_6144x16384_s1": 1003,
                     "mxfp4_experts_E256_D6144_F2048_s1_k8": 1004, "int4_g32_experts_E256_D6144_F2048_s8_k8": 1005}
    a, b = synth.workload("int4_g32_16384x6144_s1"), synth.workload("int4_g32_16384x6144_s4")
    assert a.x_key != b.x_key
    assert not np.array_equal(a.x()[0], b.x()[0])


def test_draws_are_reproducible_and_streams_independent():
    wl = synth.workload("int8_row_1024x1024_s1")
    w0, s0 = wl.weights()
    w0b, s0b = wl.weights(copy=0)
    w1, s1 = wl.weights(copy=1)
    assert np.array_equal(w0, w0b) and np.array_equal(s0, s0b)
    assert not np.array_equal(w0, w1) and not np.array_equal(s0, s1)
    ex = synth.workload("int4_g32_experts_E256_D6144_F2048_s8_k8")
    r0, r1 = ex.routing(step=0), ex.routing(step=1)
    assert np.array_equal(r0[0], ex.routing(step=0)[0])
    assert not np.array_equal(r0[0], r1[0])
    assert not np.array_equal(ex.x(step=0), ex.x(step=1))
    g0, _ = ex.expert_matrix(3, ex.GATE)
    u0, _ = ex.expert_matrix(3, ex.UP)
    g1, _ = ex.expert_matrix(4, ex.GATE)
    assert not np.array_equal(g0, u0) and not np.array_equal(g0, g1)


def test_int8_codes_cover_the_symmetric_range():
    w = synth.draw_packed(synth.INT8_ROW, 256, 4096, synth.generator(1)).view(np.int8)
    assert w.min() == -127 and w.max() == 127
    counts = np.bincount(w.astype(np.int64) + 127, minlength=255)
    assert counts.min() > 0.8 * counts.mean() and counts.max() < 1.2 * counts.mean()


@pytest.mark.parametrize("fmt", [synth.INT4_G, synth.MXFP4_G32, synth.INT3_G64])
def test_packed_codes_are_uniform(fmt):
    """Every 4-bit nibble, 2-bit pair and single bit of a packed buffer is uniform."""
    b = synth.draw_packed(fmt, 512, 4096, synth.generator(2, fmt))
    assert b.dtype == np.uint8 and b.size == synth.packed_bytes(fmt, 512, 4096)
    nib = np.concatenate([b & 15, b >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.max() < 1.05 * counts.mean() and counts.min() > 0.95 * counts.mean()
    bits = np.unpackbits(b)
    assert abs(bits.mean() - 0.5) < 0.005


def test_lognormal_scales_have_the_stated_law():
    sc = synth.draw_scales(4096, 4096, 32, synth.generator(3), "lognormal", -4.0)
    assert sc.dtype == np.float32 and sc.size == 4096 * 128 and (sc > 0).all()
    z = np.log(sc.astype(np.float64))
    assert abs(z.mean() + 4.0) < 0.01 and abs(z.std() - 0.5) < 0.01


def test_pow2_scales_are_powers_of_two_from_2m8_to_1():
    sc = synth.draw_scales(1024, 1024, 32, synth.generator(4), "pow2")
    m, e = np.frexp(sc)
    assert (m == 0.5).all()
    k = e.astype(np.int64) - 1
    assert k.min() == -8 and k.max() == 0
    assert len(np.unique(k)) == 9


def test_e8m0_expert_workload_holds_the_f32_workload_values():
    """Same seed and exponent draws: byte = 127 + log2(the f32 scale), codes identical."""
    a = synth.workload("mxfp4_experts_E256_D6144_F2048_s1_k8")
    b = synth.workload("mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8")
    for e in (0, 17, 255):
        for which in (a.GATE, a.UP, a.DOWN):
            wa, sa = a.expert_matrix(e, which)
            wb, sb = b.expert_matrix(e, which)
            assert np.array_equal(wa, wb)
            assert sb.dtype == np.uint8 and sa.dtype == np.float32
            assert np.array_equal(sb.astype(np.float64) - 127.0, np.log2(sa.astype(np.float64)))


def test_routing_law():
    """k distinct experts in [0, E) per token; weights a softmax (positive, summing to 1)."""
    wl = synth.workload("int4_g32_experts_E256_D6144_F2048_s8_k8")
    for step in range(4):
        ids, w = wl.routing(step)
        assert ids.shape == (wl.s, wl.k) and ids.dtype == np.int32
        assert w.shape == (wl.s, wl.k) and w.dtype == np.float32
        assert ids.min() >= 0 and ids.max() < wl.E
        assert all(len(set(row.tolist())) == wl.k for row in ids)
        assert (w > 0).all() and np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    lg = wl.router_logits(step=0)
    assert lg.shape == (wl.s, wl.E) and lg.dtype == np.float32


def test_compact_store_holds_exactly_the_chosen_experts():
    """store([5, 3]) = expert 5's matrices then expert 3's, for each of gate, up, down."""
    wl = synth.workload("int4_g32_experts_E256_D6144_F2048_s8_k8")
    st = wl.store([5, 3])
    for name, which in wl.MATRICES:
        nb, ns = wl.sizes(which)
        for slot, e in enumerate((5, 3)):
            w, sc = wl.expert_matrix(e, which)
            assert np.array_equal(st[name][slot * nb:(slot + 1) * nb], w)
            assert np.array_equal(st[name + "_s"][slot * ns:(slot + 1) * ns], sc)


@pytest.mark.parametrize("name,nbytes", [
    ("int8_row_1024x1024_s1", 1_052_672),
    ("int4_g32_16384x6144_s1", 62_914_560),
    ("int4_g32_16384x6144_s4", 62_914_560),
    ("int3_g64_6144x16384_s1", 44_040_192),
    ("int4_row_16384x6144_s1", 50_397_184),
    ("int8_g64_16384x6144_s1", 106_954_752),
    ("int4_g32_16384x6144_s512_prefill", 62_914_560),
])
def test_algorithmic_bytes_per_call(name, nbytes):
    """Packed codes plus scales of one call: the roofline's numerator."""
    wl = synth.workload(name)
    assert wl.weight_bytes + wl.scale_bytes == nbytes
    w, sc = wl.weights()
    assert w.nbytes + sc.nbytes == nbytes


@pytest.mark.parametrize("name,per_expert", [("mxfp4_experts_E256_D6144_F2048_s1_k8", 23_592_960),
                                             ("int4_g32_experts_E256_D6144_F2048_s8_k8", 23_592_960),
                                             ("mxfp4_e8m0_experts_E256_D6144_F2048_s1_k8", 20_054_016)])
def test_algorithmic_bytes_per_expert(name, per_expert):
    wl = synth.workload(name)
    assert wl.expert_bytes() == per_expert
    assert sum(sum(a.nbytes for a in wl.expert_matrix(0, which)) for which in (wl.GATE, wl.UP, wl.DOWN)) \
        == per_expert
