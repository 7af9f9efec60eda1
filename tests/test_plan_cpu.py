"""The fused kernel's host-side planner through nm_mlp_plan, on the CPU:
the plans of the benchmark networks, and invariants every plan must hold
(shared memory within the limit, tensor memory within 512 columns, the
thread count the roles add up to) over a seeded sweep of networks."""
import numpy as np
import pytest

from mlp_neural_gb300 import synth


@pytest.fixture(scope="module")
def nmlib():
    from mlp_neural_gb300 import build, nm
    build.build()
    return nm


@pytest.mark.parametrize("name,slots,warps,streamed,a_k", [
    ("tiny", 5, 4, 0, 32), ("page", 5, 4, 0, 64), ("wide", 3, 4, 1, 64), ("hetero", 1, 16, 1, 256)])
def test_benchmark_network_plans(nmlib, name, slots, warps, streamed, a_k):
    # wide: three slots of 160 TMEM columns (128 for the accumulator, 32 for
    # the first 64 columns of A), the other 64 columns of A in shared memory
    p = nmlib.plan(synth.WORKLOADS[name].dims)
    assert (p["tile_slots"], p["warps_per_slot"], p["streamed_weights"]) == (slots, warps, streamed)
    assert p["a_tmem_k"] == a_k
    assert p["threads"] == _threads(slots, warps, streamed)
    assert p["weight_stages"] == (4 if streamed else 0)
    assert p["smem_bytes"] <= nmlib.GB300_SMEM_OPTIN and p["tmem_columns"] == 512


def _threads(slots, warps, streamed):
    # streamed weights: the slots' warps, a weight producer and an input
    # producer; resident weights: eight warps for the slots' issuing warps
    # and the input producer, then the slots' epilogue warps
    return 32 * (slots * warps + 2) if streamed else 32 * (8 + slots * warps)


def _tmem_needed(dims, slots, per_col=2, a_k=256):
    # per slot: the FP32 accumulator of the widest layer and the next layer's
    # A for the widest hidden layer, as far as it is kept in TMEM (FP16 pairs,
    # or E4M3 quads for the narrow-precision variant; each rounded up to 32
    # columns), plus one 32-column block for the shared ones slab
    r32 = lambda c: (c + 31) // 32 * 32
    acc = r32(max(dims[1:]))
    hidden = min(a_k, max([16] + list(dims[1:-1])))
    return slots * (acc + r32(hidden // per_col)) + 32


@pytest.mark.parametrize("name,slots,warps", [("wide", 3, 4), ("hetero", 1, 16), ("page", 3, 4)])
def test_fp8_plans_stream_their_weights(nmlib, name, slots, warps):
    p = nmlib.plan(synth.WORKLOADS[name].dims, nmlib.NM_VARIANT_FP8_WEIGHTS)
    assert (p["tile_slots"], p["warps_per_slot"], p["streamed_weights"]) == (slots, warps, 1)
    assert p["threads"] == _threads(slots, warps, 1)


@pytest.mark.parametrize("dims", [(32, 16), (32, 48, 16), (64, 128, 80, 16)])
def test_fp8_plan_needs_e4m3_images(nmlib, dims):
    with pytest.raises(nmlib.NmError) as e:
        nmlib.plan(dims, nmlib.NM_VARIANT_FP8_WEIGHTS)
    assert e.value.status == nmlib.NM_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,fused_issuers,paired_issuers", [
    ("tiny", 5, 3), ("page", 5, 3), ("wide", 3, 3), ("hetero", 1, 1)])
def test_issuing_warps(nmlib, name, fused_issuers, paired_issuers):
    # one issuing warp per tile slot; the paired-tiles variant issues the
    # resident-weight slots two at a time (2 + 2 + 1 for five slots)
    dims = synth.WORKLOADS[name].dims
    assert nmlib.plan(dims)["issuing_warps"] == fused_issuers
    p = nmlib.plan(dims, nmlib.NM_VARIANT_PAIRED_TILES)
    assert p["issuing_warps"] == paired_issuers
    assert p["tile_slots"] == nmlib.plan(dims)["tile_slots"]


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_plan_invariants_over_random_networks(nmlib, variant):
    rng = np.random.default_rng(100 + variant)
    planned = 0
    for _ in range(400):
        L = int(rng.integers(1, 17))
        dims = [int(16 * rng.integers(1, 17)) for _ in range(L + 1)]
        if variant == 4:  # hidden widths that have E4M3 images
            L = max(L, 2)
            dims = ([int(16 * rng.integers(1, 17))] + [int(32 * rng.integers(1, 9)) for _ in range(L - 1)]
                    + [int(16 * rng.integers(1, 17))])
        try:
            p = nmlib.plan(dims, variant)
        except nmlib.NmError as e:
            assert e.status == nmlib.NM_ERR_UNSUPPORTED
            continue
        planned += 1
        slots, warps = p["tile_slots"], p["warps_per_slot"]
        assert 1 <= slots <= 5 and warps % 4 == 0
        assert p["threads"] == _threads(slots, warps, p["streamed_weights"]) <= 1024
        assert p["smem_bytes"] <= nmlib.GB300_SMEM_OPTIN
        t = p["tmem_columns"]
        assert 32 <= t <= 512 and t & (t - 1) == 0
        assert _tmem_needed(dims, slots, 4 if variant == 4 else 2, p["a_tmem_k"]) <= t
        hidden = max([16] + list(dims[1:-1]))
        if p["a_tmem_k"] < hidden:
            # split A: streamed FP16 only, whole 64-column segments in smem
            assert p["streamed_weights"] and variant in (0, 3)
            assert p["a_tmem_k"] % 64 == 0
            assert all(d <= p["a_tmem_k"] or d % 64 == 0 for d in dims[1:-1])
            assert _tmem_needed(dims, slots) > 512
        assert p["input_stages"] in (1, 2) and p["output_buffers"] in (1, 2)
        if p["streamed_weights"]:
            assert variant != 1 and slots <= 3 and 2 <= p["weight_stages"] <= 4
            if variant == 4:
                assert all(d % 32 == 0 for d in dims[1:-1]) and L >= 2
            assert p["issuing_warps"] == slots
        else:
            assert variant != 4 and p["weight_stages"] == 0
            paired = variant == 3 and warps == 4
            assert p["issuing_warps"] == ((slots + 1) // 2 if paired else slots)
    assert planned > 200


def test_split_a_only_for_whole_segments(nmlib):
    # 112-wide hidden layers leave a 48-column remainder: no split, 2 slots
    p = nmlib.plan((80,) + (112,) * 8 + (16,))
    assert (p["tile_slots"], p["a_tmem_k"]) == (2, 112)
    # 64- and 128-wide hidden layers: the 64-wide ones wholly in TMEM
    p = nmlib.plan((128, 128, 64, 128, 128, 128, 128, 64, 128, 16))
    assert (p["tile_slots"], p["a_tmem_k"], p["streamed_weights"]) == (3, 64, 1)


def test_three_streamed_slots(nmlib):
    # 160 TMEM columns a slot (96 accumulator + 64 for the FP16 A of a
    # 96-wide layer): three slots of one column group each
    p = nmlib.plan((64,) + (96,) * 15 + (16,))
    assert (p["tile_slots"], p["warps_per_slot"], p["streamed_weights"]) == (3, 4, 1)


def test_smaller_shared_memory_limit_gives_a_smaller_plan(nmlib):
    dims = synth.WORKLOADS["page"].dims
    big = nmlib.plan(dims)
    small = nmlib.plan(dims, smem_optin=100 * 1024)
    assert small["smem_bytes"] <= 100 * 1024
    assert small["tile_slots"] <= big["tile_slots"]


def test_plan_argument_errors(nmlib):
    with pytest.raises(nmlib.NmError) as e:
        nmlib.plan((32, 24))
    assert e.value.status == nmlib.NM_ERR_UNSUPPORTED
    with pytest.raises(nmlib.NmError) as e:
        nmlib.plan((32, 16), variant=7)
    assert e.value.status == nmlib.NM_ERR_INVALID_ARG
    with pytest.raises(nmlib.NmError) as e:
        nmlib.plan((32,))
    assert e.value.status == nmlib.NM_ERR_INVALID_ARG
