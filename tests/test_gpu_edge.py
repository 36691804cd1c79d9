"""Edge cases of the GPU verifier, each checked against the oracle or the
documented status bits."""
import numpy as np
import pytest

import oracle
import synth
from parity import assert_parity, check_structure, compare, run_gpu

pytestmark = pytest.mark.gpu


def make_batch(logits, gammas, ids, temps, q=None, top_k=None, top_p=None, dtype="f32", seed=3,
               flags=0):
    gammas = np.asarray(gammas, np.int32)
    B = gammas.size
    cu = np.zeros(B + 1, np.int32)
    np.cumsum(gammas, out=cu[1:])
    logits = np.asarray(logits, np.float32)
    if dtype == "bf16":
        logits = synth.f32_to_bf16_bits(logits)
    return dict(B=B, V=logits.shape[1], cu_num_draft=cu,
                draft_token_ids=np.asarray(ids, np.int32).reshape(-1),
                target_logits=logits, logits_dtype=dtype,
                draft_probs=None if q is None else np.asarray(q, np.float32),
                temperature=np.asarray(temps, np.float32),
                top_k=None if top_k is None else np.asarray(top_k, np.int32),
                top_p=None if top_p is None else np.asarray(top_p, np.float32),
                seed=seed, request_base=0, flags=flags)


def random_case(seed, B=40, V=300, gmax=6, dtype="f32", prob=True, ties=False):
    rng = np.random.default_rng(seed)
    g = rng.integers(0, gmax + 1, size=B)
    N = int(g.sum())
    logits = rng.normal(0, 2, size=(N + B, V))
    if ties:
        logits = np.round(logits)
    q = rng.random((N, V)) ** 3
    q /= q.sum(1, keepdims=True)
    ids = np.array([rng.choice(V, p=q[n]) for n in range(N)], np.int32)
    temps = rng.choice([0.0, 0.01, 0.5, 1.0, 3.0, 100.0], size=B)
    tk = rng.choice([0, 1, 2, 7, V, V + 5], size=B)
    tp = rng.choice([1.0, 0.001, 0.5, 0.9, 0.99], size=B)
    return make_batch(logits, g, ids, temps, q if prob else None, tk, tp, dtype=dtype, seed=seed)


def check(b, greedy=False):
    gpu = run_gpu(b, greedy=greedy)
    ref = oracle.verify(b)
    check_structure(b, gpu)
    assert_parity(compare(b, gpu, ref))
    return gpu, ref


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("prob", [True, False])
def test_random_mixed_settings(seed, dtype, prob):
    gpu, _ = check(random_case(seed, dtype=dtype, prob=prob, ties=seed % 2 == 1))
    assert gpu["status"] & ~np.uint32(0x8) == 0


def test_empty_batch():
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    ver = sv.Verifier(max_batch=4, max_rows=8, max_vocab=16)
    dev = "cuda:0"
    db = sv.DeviceBatch(cu_num_draft=torch.zeros(1, dtype=torch.int32, device=dev),
                        draft_token_ids=torch.zeros(0, dtype=torch.int32, device=dev),
                        target_logits=torch.zeros(0, 16, device=dev), draft_probs=None,
                        temperature=torch.zeros(0, device=dev), N=0, V=16)
    ver.run(db)
    ver.greedy(db)
    torch.cuda.synchronize()
    assert ver.status() == 0
    ver.close()


def test_no_draft_tokens_bonus_only():
    b = random_case(1, B=50, gmax=0)
    assert int(b["cu_num_draft"][-1]) == 0
    check(b)


def test_single_token_vocabulary():
    b = random_case(2, B=20, V=1)
    gpu, _ = check(b)
    assert np.all(gpu["out_tokens"][gpu["out_tokens"] >= 0] == 0)


def test_long_rounds():
    check(random_case(3, B=12, gmax=40, V=500))


def test_minus_inf_logits():
    rng = np.random.default_rng(4)
    b = random_case(4, B=30, V=64)
    logits = b["target_logits"]
    logits[rng.random(logits.shape) < 0.7] = -np.inf
    logits[:, 5] = 0.25  # every row keeps one finite logit
    check(b)


def test_uniform_rows_and_top_p():
    b = random_case(5, B=30, V=100, dtype="bf16")
    b["target_logits"][:] = synth.f32_to_bf16_bits(np.float32(1.5))
    check(b)


def test_invalid_token_ids_set_status():
    b = random_case(6, B=30, V=80)
    ids = b["draft_token_ids"]
    ids[::5] = -1
    ids[1::7] = 80
    gpu, ref = check(b)
    assert gpu["status"] & 0x4


def test_nonfinite_rows_set_status():
    b = random_case(7, B=30, V=80)
    b["temperature"][:] = 1.0
    b["target_logits"][3, 10] = np.nan
    b["target_logits"][9, 1] = np.inf
    gpu = run_gpu(b)
    ref = oracle.verify(b)
    assert gpu["status"] & 0x1
    bad = (ref["req_status"] & 1) != 0
    assert bad.sum() >= 1
    for r in np.nonzero(bad)[0]:
        assert gpu["num_accepted"][r] == 0
    assert_parity(compare(b, gpu, ref, requests=np.nonzero(~bad)[0]))


def test_bad_offsets_set_status():
    b = random_case(8, B=6, V=50)
    cu = b["cu_num_draft"].copy()
    cu[2], cu[3] = cu[3], cu[2] - 1 if cu[2] > 0 else 0
    b["cu_num_draft"] = cu
    gpu = run_gpu(b)
    assert gpu["status"] & 0x10


def test_temperature_zero_ignores_draft_probs():
    b = random_case(9, B=40, V=200)
    b["temperature"][:] = 0
    b["draft_probs"][:] = 0  # must never be read at temperature 0
    check(b)


@pytest.mark.parametrize("scale", [0.01, 0.2, 2.0, 30.0, 400.0, "ties"])
@pytest.mark.parametrize("V", [304, 4096])
def test_filtered_rows_on_the_streaming_path(scale, V):
    """Aligned bf16 rows with top-k / top-p take the histogram path of the
    streaming pass; tiny logits (threshold near 0) and |l| >= 256 fall back
    to the exact search. Both must agree with the oracle."""
    rng = np.random.default_rng(V + (7 if scale == "ties" else int(float(scale) * 100)))
    B = 36
    g = rng.integers(0, 5, size=B)
    N = int(g.sum())
    if scale == "ties":
        logits = np.round(rng.normal(0, 2, size=(N + B, V)))
    else:
        logits = rng.normal(0, float(scale), size=(N + B, V))
    q = rng.random((N, V)) ** 2
    q /= q.sum(1, keepdims=True)
    ids = np.array([rng.choice(V, p=q[n]) for n in range(N)], np.int32)
    temps = rng.choice([0.0, 0.5, 1.0, 2.0], size=B)
    tk = rng.choice([0, 1, 5, 50, V], size=B)
    tp = rng.choice([1.0, 0.3, 0.9, 0.999], size=B)
    b = make_batch(logits, g, ids, temps, q, tk, tp, dtype="bf16", seed=V)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


@pytest.mark.parametrize("case", ["wide_top_k", "tiny_temperature", "both_filters", "heavy_tail"])
def test_window_histogram_cases(case):
    """Regimes of the window histogram of the filtered row pass: top-k sets
    reaching past the window (left to the exact slow kernel), narrow windows
    at small temperature, top-k and top-p together, and a top-p boundary on
    a value that thousands of tokens share."""
    rng = np.random.default_rng(["wide_top_k", "tiny_temperature", "both_filters",
                                 "heavy_tail"].index(case) + 91)
    V, B = 4096, 30
    g = rng.integers(0, 4, size=B)
    N = int(g.sum())
    tk = tp = None
    if case == "wide_top_k":
        logits = rng.normal(0, 15, size=(N + B, V))
        temps = rng.choice([0.5, 1.0], size=B)
        tk = rng.choice([1000, 3000, 4000], size=B)
    elif case == "tiny_temperature":
        logits = rng.normal(0, 2, size=(N + B, V))
        temps = rng.choice([0.01, 0.05], size=B)
        tp = rng.choice([0.5, 0.9, 0.999], size=B)
    elif case == "both_filters":
        logits = rng.normal(0, 3, size=(N + B, V))
        temps = np.ones(B)
        tk = rng.choice([20, 200], size=B)
        tp = rng.choice([0.5, 0.95], size=B)
    else:
        logits = np.full((N + B, V), -5.0)
        hot = rng.integers(0, V, size=(N + B, 40))
        for r in range(N + B):
            logits[r, hot[r]] = rng.uniform(-1, 3, size=40)
        temps = np.ones(B)
        tp = rng.choice([0.5, 0.9, 0.99], size=B)
    q = rng.random((N, V)) ** 2
    q /= q.sum(1, keepdims=True)
    ids = np.array([rng.choice(V, p=q[n]) for n in range(N)], np.int32)
    b = make_batch(logits, g, ids, temps, q, tk, tp, dtype="bf16", seed=17)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


@pytest.mark.parametrize("case", ["tiny_kept", "tiny_boundary"])
def test_window_histogram_tiny_magnitudes(case):
    """Rows whose counted values include many magnitudes below 2^-16 (and
    exact zeros of both signs), at temperatures where their weights differ
    visibly from one another: their exact weight sums must reach Z and the
    kept mass whether the top-p boundary lies above them ("tiny_kept") or
    among them ("tiny_boundary", left to the exact slow kernel)."""
    rng = np.random.default_rng(["tiny_kept", "tiny_boundary"].index(case) + 301)
    V, B = 4096, 24
    g = rng.integers(0, 4, size=B)
    N = int(g.sum())
    logits = rng.normal(0, 6e-6, size=(N + B, V))
    logits[rng.random((N + B, V)) < 0.1] = 0.0
    logits[rng.random((N + B, V)) < 0.05] = -0.0
    if case == "tiny_kept":
        # a few heavier tokens put the boundary above the tiny values, or
        # keep all of them when top_p is high
        hot = rng.integers(0, V, size=(N + B, 30))
        for r in range(N + B):
            logits[r, hot[r]] = rng.uniform(0.0005, 0.004, size=30)
        temps = rng.choice([0.0005, 0.001], size=B)
        tp = rng.choice([0.3, 0.9, 0.9999], size=B)
    else:
        temps = rng.choice([0.00002, 0.0001], size=B)
        tp = rng.choice([0.5, 0.9], size=B)
    q = rng.random((N, V)) ** 2
    q /= q.sum(1, keepdims=True)
    ids = np.array([rng.choice(V, p=q[n]) for n in range(N)], np.int32)
    b = make_batch(logits, g, ids, temps, q, None, tp, dtype="bf16", seed=29)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


def test_bounded_wait_times_out_and_the_context_survives():
    """A wait that cannot be satisfied ends with SPEC_STATUS_TIMEOUT instead
    of hanging: a test-only handle flag leaves the early-exit work queue
    empty (nothing will ever fill the slots the readers wait on) and gives
    those waits a few polls. The same process then verifies a batch
    correctly with a normal handle."""
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    b = synth.make("c5", B=16, V=20000)
    b["flags"] = sv.FLAG_EARLY_EXIT
    R = b["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=16, max_rows=R, max_vocab=20000,
                      config_flags=sv.CONFIG_TEST_WAIT_TIMEOUT | sv.CONFIG_EARLY_QUEUE)
    db = sv.upload(b, "cuda:0")
    ver.run(db)
    torch.cuda.synchronize()
    assert ver.status() & sv.STATUS_TIMEOUT
    ver.close()
    gpu, _ = check(b)
    assert gpu["status"] == 0


TOP_P_CASES = ["late_max", "one_far_logit", "masked_first_stage", "flat_rows", "tiny_top_p",
               "wide_top_p", "far_negative"]


@pytest.mark.parametrize("case", TOP_P_CASES)
def test_top_p_only_multi_stage_cases(case):
    """Top-p without top-k on aligned bf16 rows of several 12288-element
    stages of the filtered row pass: the row max far above the first
    stage's, one logit far above the rest, a first stage of -inf only, rows
    of one or two values, top-p sets of one token and of nearly the whole
    row, and logits far below zero."""
    rng = np.random.default_rng(TOP_P_CASES.index(case) + 301)
    V, B = 37864, 12
    g = rng.integers(0, 4, size=B)
    N = int(g.sum())
    R = N + B
    temps = rng.choice([0.5, 1.0, 2.0], size=B)
    tp = rng.choice([0.3, 0.9, 0.99], size=B)
    logits = rng.normal(0, 2, size=(R, V))
    if case == "late_max":
        cols = 20000 + rng.integers(0, 17000, size=R)
        logits[np.arange(R), cols] = 20.0
        logits[: R // 2, cols[0] // 2 + 14000] = 12.0
    elif case == "one_far_logit":
        logits[:, :12288] = rng.normal(0, 0.5, size=(R, 12288))
        logits[np.arange(R), 25000 + rng.integers(0, 12000, size=R)] = 150.0
        temps = np.full(B, 0.5)
    elif case == "masked_first_stage":
        logits[:, :13000] = -np.inf
    elif case == "flat_rows":
        logits[:] = 0.75
        logits[::3, ::7] = 0.5
    elif case == "tiny_top_p":
        tp = np.full(B, 0.001)
    elif case == "wide_top_p":
        logits = rng.normal(0, 6, size=(R, V))
        tp = rng.choice([0.999, 0.99999], size=B)
    else:
        logits = rng.normal(-180, 3, size=(R, V))
        temps = rng.choice([0.25, 1.0], size=B)
    q = rng.random((N, V)) ** 2
    q /= q.sum(1, keepdims=True)
    ids = np.array([rng.choice(V, p=q[n]) for n in range(N)], np.int32)
    b = make_batch(logits, g, ids, temps, q, None, tp, dtype="bf16", seed=29)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


@pytest.mark.parametrize("schedule", ["full", "queue", "resident"])
@pytest.mark.parametrize("V,dtype", [(300, "f32"), (20008, "bf16"), (20011, "bf16")])
def test_all_residual_weights_zero_draw_from_p(V, dtype, schedule):
    """Draft probabilities of 1 at every token: after a rejection every
    residual weight max(p - q, 0) is 0, so the token is drawn from p over the
    whole row and the empty-residual status bit is set, as the oracle reads
    a residual of zero mass. V = 20011 bf16 rows are not 16-byte aligned (the
    race reads them from global memory)."""
    import speculative_decoding_rejection_02_gb300 as sv
    rng = np.random.default_rng(11)
    B = 24
    g = rng.integers(1, 5, size=B)
    N = int(g.sum())
    logits = rng.normal(0, 2, size=(N + B, V))
    q = np.ones((N, V), np.float32)
    ids = rng.integers(0, V, size=N).astype(np.int32)
    early = schedule != "full"
    b = make_batch(logits, g, ids, np.ones(B, np.float32), q, dtype=dtype, seed=7,
                   flags=sv.FLAG_EARLY_EXIT if early else 0)
    config = {"full": 0, "queue": sv.CONFIG_EARLY_QUEUE,
              "resident": sv.CONFIG_EARLY_RESIDENT}[schedule]
    ver = sv.Verifier(max_batch=B, max_rows=N + B, max_vocab=V, config_flags=config)
    try:
        gpu = run_gpu(b, verifier=ver)
    finally:
        ver.close()
    ref = oracle.verify(b)
    check_structure(b, gpu)
    assert_parity(compare(b, gpu, ref))
    empty = (ref["req_status"] & 0x8) != 0
    assert empty.sum() >= B // 2
    assert gpu["status"] & 0x8
    assert gpu["status"] & ~np.uint32(0x8) == 0


def test_masked_races_repeat_exactly():
    """Every draft token is its row's argmax and one-hot, so each rejection
    races with the argmax masked and no seeded best: the race's first slice
    starts from its own heaviest entry while later slices publish theirs.
    Sixteen calls must all give the oracle's tokens (a block that disagreed
    about its starting best once paired a weight with the wrong index)."""
    rng = np.random.default_rng(404)
    V, B = 131072, 256
    g = np.ones(B, np.int32)
    logits = rng.normal(0, 2, size=(2 * B, V)).astype(np.float32)
    ids = np.argmax(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(logits))[0::2], axis=1)
    b = make_batch(logits, g, ids.astype(np.int32), np.ones(B), dtype="bf16", seed=41)
    ref = oracle.verify(b)
    for _ in range(16):
        gpu = run_gpu(b)
        assert_parity(compare(b, gpu, ref))


@pytest.mark.parametrize("name,B,V", [("c2", 8, 32000), ("c3", 24, 20008), ("c3", 24, 20011),
                                      ("c5", 40, 20008)])
def test_draft_probs_in_page_locked_host_memory(name, B, V):
    """draft_probs left in page-locked host memory is read in place: the same
    outputs as with the rows on the device, and parity with the oracle."""
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    batch = synth.make(name, B=B, V=V)
    R = batch["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=B, max_rows=R, max_vocab=V)
    on_dev = sv.upload(batch, "cuda:0")
    ver.run(on_dev)
    on_host = sv.upload(batch, "cuda:0")
    on_host.draft_probs = torch.from_numpy(batch["draft_probs"]).pin_memory()
    ver.run(on_host)
    torch.cuda.synchronize()
    assert ver.status() == 0
    assert torch.equal(on_dev.num_accepted, on_host.num_accepted)
    assert torch.equal(on_dev.out_tokens, on_host.out_tokens)
    assert torch.equal(on_dev.p_at_draft, on_host.p_at_draft)
    gpu = dict(out_tokens=on_host.out_tokens.cpu().numpy(),
               num_accepted=on_host.num_accepted.cpu().numpy(),
               p_at_draft=on_host.p_at_draft.cpu().numpy(), status=0)
    assert_parity(compare(batch, gpu, oracle.verify(batch)))
    ver.close()


def test_pageable_draft_probs_are_rejected():
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    batch = synth.make("c2", B=2, V=64)
    R = batch["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=2, max_rows=R, max_vocab=64)
    db = sv.upload(batch, "cuda:0")
    db.draft_probs = torch.from_numpy(batch["draft_probs"])  # not page-locked
    with pytest.raises(sv.SpecVerifyError) as err:
        ver.run(db)
    assert err.value.code == -1
    ver.close()


def test_draft_probs_in_host_memory_under_early_exit():
    """Early exit through its work queue (the row pass judges positions and
    gathers q(x) itself) with draft_probs left in page-locked host memory:
    the same outputs as with the rows on the device."""
    import torch

    import speculative_decoding_rejection_02_gb300 as sv
    batch = synth.make("c5", B=40, V=20008)
    batch["flags"] = sv.FLAG_EARLY_EXIT
    R = batch["target_logits"].shape[0]
    ver = sv.Verifier(max_batch=40, max_rows=R, max_vocab=20008,
                      config_flags=sv.CONFIG_EARLY_QUEUE)
    on_dev = sv.upload(batch, "cuda:0")
    ver.run(on_dev)
    on_host = sv.upload(batch, "cuda:0")
    on_host.draft_probs = torch.from_numpy(batch["draft_probs"]).pin_memory()
    ver.run(on_host)
    torch.cuda.synchronize()
    assert ver.status() == 0
    assert torch.equal(on_dev.num_accepted, on_host.num_accepted)
    assert torch.equal(on_dev.out_tokens, on_host.out_tokens)
    ver.close()


@pytest.mark.parametrize("V", [32000, 32001])
def test_fp32_rows_with_top_k_and_top_p(V):
    """fp32 target rows with top-k and top-p have no window histogram: the
    exact kernel settles them by radix selection over 32-bit keys (four
    8-bit digits), aligned and misaligned rows, ties included."""
    b = synth.make("c2", B=24, V=V)
    rng = np.random.default_rng(V)
    logits = b["target_logits"].copy()
    logits[::3] = np.round(logits[::3] * 2) / 2  # rows of tied values
    b["target_logits"] = logits
    b["top_k"] = rng.choice([0, 1, 7, 50, 3000], size=b["B"]).astype(np.int32)
    b["top_p"] = rng.choice([1.0, 0.3, 0.9, 0.99], size=b["B"]).astype(np.float32)
    b["temperature"] = rng.choice([0.0, 0.5, 1.0, 2.0], size=b["B"]).astype(np.float32)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


@pytest.mark.parametrize("mode", ["top_p", "top_k", "both"])
def test_fp32_single_filters_at_a_large_vocabulary(mode):
    """fp32 rows at V = 151936 with top-p only, top-k only, or both: the
    first two settled from the histogram of truncated values (wide candidate
    ranges near the boundary), the third by the exact search."""
    b = synth.make("c2", B=6, V=151936)
    rng = np.random.default_rng(17)
    B = b["B"]
    b["temperature"] = rng.choice([0.5, 1.0, 2.0], size=B).astype(np.float32)
    if mode in ("top_p", "both"):
        b["top_p"] = rng.choice([0.3, 0.9, 0.99], size=B).astype(np.float32)
    if mode in ("top_k", "both"):
        b["top_k"] = rng.choice([1, 50, 20000], size=B).astype(np.int32)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0


def test_fp32_flat_rows_overflow_the_candidate_buffer():
    """fp32 rows whose values all sit in a few bf16-truncated bins: the bins
    around the top-p boundary hold more values than the select kernel's
    buffer, so those rows take the exact search in the same block."""
    b = synth.make("c2", B=4, V=60000)
    rng = np.random.default_rng(23)
    R = b["target_logits"].shape[0]
    b["target_logits"] = (1.0 + rng.normal(0, 1e-3, size=(R, b["V"]))).astype(np.float32)
    b["top_p"] = np.full(b["B"], 0.5, np.float32)
    gpu, _ = check(b)
    assert gpu["status"] & ~np.uint32(0x8) == 0
