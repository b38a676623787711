"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by
element on identical seeded inputs.

Small sizes compare every element (they span several blocks' tiles and a
ragged tail); so do the full-size HBM workloads, whose oracle runs over the
whole unit (its functions on disjoint slices in threads, the clip norm over
the whole mean gradient).

Gate: |gpu - oracle| <= 2e-6*(1+|oracle|) on FP32 master, m, v after every
step, and <= 1 BF16 ulp on the emitted copy.  Without the clip the two
follow the same FP32 operation sequence, so those cases also require bit
equality.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import workloads as W  # noqa: E402
import parity_util as pu  # noqa: E402


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


def dev_u16(n):
    return torch.empty(max(n, 1) + 64, dtype=torch.int16, device="cuda")


def dev_grad_buf(n, fp32=False):
    """Device buffer for one gradient replica of n values (BF16 or FP32)."""
    return torch.empty(max(n, 1) + 64, dtype=torch.float32 if fp32 else torch.int16, device="cuda")


def to_np_u16(t, n):
    return t[:n].cpu().numpy().view(np.uint16)


# -------------------------------------------------------------- generator ----

def test_generator_device_matches_host(S):
    n, off = (1 << 20) + 3, 12345
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.dev_master(out.data_ptr(), n, seed=9, unit=3, scale=0.02, offset=off)
    torch.cuda.synchronize()
    host = synth.master(n, seed=9, unit=3, scale=0.02, offset=off)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), host.view(np.uint32))
    for kind, zp in ((synth.GRAD_NORMAL, 0.0), (synth.GRAD_STUDENT3, 0.001)):
        sp = synth.spec(5, kind, zp)
        g = dev_u16(n)
        synth.dev_grad(g.data_ptr(), n, sp, 2, 7, 3, 1e-3, offset=off)
        torch.cuda.synchronize()
        assert np.array_equal(to_np_u16(g, n), synth.grad(n, sp, 2, 7, 3, 1e-3, offset=off))


# ------------------------------------------------------ small, every element ----

def run_small(S, sizes, R, clip, steps=4, seed=11, flags=0, bf16_external=False, fp32=False):
    """Multi-layer state with the given layer sizes; `steps` steps of every
    layer on fresh seeded grads; full comparison with the oracle after each."""
    w = W.Workload("small", [W.Unit(f"l{i}", [("flat", n)]) for i, n in enumerate(sizes)],
                   R=R, steps=steps, seed=seed, max_grad_norm=clip, lr=1e-3, fp32_grads=fp32)
    if fp32:
        flags |= S.SLIDE_FLAG_FP32_GRADS
    hp_dev = S.hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_grad_norm)
    hp_or = pu.hp_oracle(w)
    st = S.slide_state_create(sizes, R, flags=flags)
    reports = []
    try:
        ref = []
        for li, n in enumerate(sizes):
            th0 = synth.master(n, seed, unit=li)
            S.slide_layer_set(st, li, master=th0, step=0)
            ref.append([th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
                        np.zeros(n, np.uint16)])
        grads = [dev_grad_buf(max(sizes), fp32) for _ in range(R)]
        outs = [dev_u16(n) for n in sizes] if bf16_external else None
        for t in range(1, steps + 1):
            for li, n in enumerate(sizes):
                for r in range(R):
                    pu.unit_grad_dev(w, li, t, r, grads[r].data_ptr())
                S.slide_layer_step(st, li, grads, hp_dev, None, outs[li] if outs else None)
                host_g = [pu.unit_grad_host(w, li, t, r) for r in range(R)]
                coef = oracle.layer_step(host_g, *ref[li][:3], ref[li][3], hp_or, t)
                th, m, v = (np.empty(n, np.float32) for _ in range(3))
                wb = np.empty(n, np.uint16)
                tt = S.slide_layer_get(st, li, th, m, v, wb)
                assert tt == t
                if bf16_external:
                    torch.cuda.synchronize()
                    wb = to_np_u16(outs[li], n)
                rep = [pu.compare_fp32(f"theta l{li} t{t}", th, ref[li][0]),
                       pu.compare_fp32(f"m l{li} t{t}", m, ref[li][1]),
                       pu.compare_fp32(f"v l{li} t{t}", v, ref[li][2]),
                       pu.compare_bf16(f"w l{li} t{t}", wb, ref[li][3])]
                pu.assert_parity(rep)
                # the emitted copy is the RNE rounding of the GPU's own master
                assert np.array_equal(wb, oracle.f32_to_bf16(th))
                if clip > 0 and n > 0:
                    gc = S.slide_layer_last_clip_coef(st, li)
                    assert abs(gc - coef) <= 2 * np.spacing(np.float32(coef)), (gc, coef)
                if flags & S.SLIDE_FLAG_CHECK_FINITE:   # finite inputs: nothing may be flagged
                    assert S.slide_layer_status(st, li) == S.SLIDE_OK
                reports += rep
    finally:
        S.slide_state_destroy(st)
    return reports


SIZES = [1, 7, 8, 9, 1000, 1001, 4096 + 3, (1 << 20) + 5]


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
def test_small_parity_no_clip_bit_exact(S, R):
    reps = run_small(S, SIZES, R, clip=0.0)
    for r in reps:
        assert r["not_bit_equal"] == 0, r


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("clip", [1e-3, 1e3])
def test_small_parity_clip(S, R, clip):
    reps = run_small(S, [9, 4096 + 3, (1 << 20) + 5, 3 * (1 << 20) + 1], R, clip=clip)
    if clip > 1.0:  # norm far below the threshold: coefficient exactly 1
        for r in reps:
            assert r["not_bit_equal"] == 0, r


@pytest.mark.parametrize("scale", [1e-8, 1e-10, 1e-30])
def test_eps_regime_bit_exact(S, scale):
    """Gradients around and far below eps (1e-8): the update is governed by
    the eps term; still the same FP32 operations on both sides."""
    n, R = 70001, 4
    w = W.Workload("eps", [W.Unit("l", [("flat", n)])], R=R, steps=4, seed=41, grad_scale=scale, lr=1e-3)
    hp_dev = S.hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, 0.0)
    hp_or = pu.hp_oracle(w)
    th = synth.master(n, w.seed)
    m, v, wb = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    st = S.slide_state_create([n], R)
    try:
        S.slide_layer_set(st, 0, master=th, step=0)
        grads = [dev_u16(n) for _ in range(R)]
        for t in range(1, 5):
            for r in range(R):
                pu.unit_grad_dev(w, 0, t, r, grads[r].data_ptr())
            S.slide_layer_step(st, 0, grads, hp_dev)
            oracle.layer_step([pu.unit_grad_host(w, 0, t, r) for r in range(R)], th, m, v, wb, hp_or, t)
        a, b, c = (np.empty(n, np.float32) for _ in range(3))
        gw = np.empty(n, np.uint16)
        S.slide_layer_get(st, 0, a, b, c, gw)
        rep = [pu.compare_fp32("theta", a, th), pu.compare_fp32("m", b, m), pu.compare_fp32("v", c, v),
               pu.compare_bf16("w", gw, wb)]
        pu.assert_parity(rep)
        assert all(r["not_bit_equal"] == 0 for r in rep), rep
    finally:
        S.slide_state_destroy(st)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
def test_small_parity_fp32_grads(S, R, clip):
    """FP32 gradient replicas (26 + 4R bytes per parameter): same arithmetic
    after the widening, so bit-exact without a clip."""
    reps = run_small(S, [1, 9, 4096 + 3, (1 << 20) + 5], R, clip=clip, fp32=True)
    if clip == 0.0:
        for r in reps:
            assert r["not_bit_equal"] == 0, r


@pytest.mark.parametrize("R,fp32", [(1, False), (4, False), (8, False), (3, True), (6, True), (8, True)])
def test_clipped_steps_back_to_back_overlapped_and_serialised(S, R, fp32):
    """Clipped steps of three layers enqueued back to back on one stream, with
    no host synchronisation between them.  A clipped step starts while its
    pre-pass still runs (where a CTA of each fits on an SM together: BF16
    replicas, and FP32 replicas up to R = 6) unless trace events sit between
    the two, as they do for the second state here.  Both states must end with
    the same bits, and with the oracle's result within the tolerance."""
    sizes = [3 * (1 << 20) + 5, 2048 * 152 * 2 + 7, 4099]
    steps = 4
    w = W.Workload("b2b", [W.Unit(f"l{i}", [("flat", n)]) for i, n in enumerate(sizes)], R=R, steps=steps,
                   seed=77, max_grad_norm=1e-3, lr=1e-3, fp32_grads=fp32)
    hp = S.hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_grad_norm)
    flags = S.SLIDE_FLAG_FP32_GRADS if fp32 else 0
    stream = torch.cuda.Stream()
    # every step's replicas are generated up front, so nothing waits between steps
    grads = {}
    for t in range(1, steps + 1):
        for li, n in enumerate(sizes):
            grads[t, li] = [dev_grad_buf(n, fp32) for _ in range(R)]
            for r in range(R):
                pu.unit_grad_dev(w, li, t, r, grads[t, li][r].data_ptr())
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize()
    overlapped = S.slide_state_create(sizes, R, flags=flags)
    serialised = S.slide_state_create(sizes, R, flags=flags)
    try:
        th0 = [synth.master(n, w.seed, unit=li) for li, n in enumerate(sizes)]
        for st in (overlapped, serialised):
            for li in range(len(sizes)):
                S.slide_layer_set(st, li, master=th0[li], step=0)
        S.slide_trace_events(serialised, *ev)
        for t in range(1, steps + 1):
            for li in range(len(sizes)):
                S.slide_layer_step(overlapped, li, grads[t, li], hp, stream)
                S.slide_layer_step(serialised, li, grads[t, li], hp, stream)
        torch.cuda.synchronize()
        S.slide_trace_events(serialised)
        hp_or = pu.hp_oracle(w)
        for li, n in enumerate(sizes):
            got = []
            for st in (overlapped, serialised):
                a, b, c = (np.empty(n, np.float32) for _ in range(3))
                wb = np.empty(n, np.uint16)
                assert S.slide_layer_get(st, li, a, b, c, wb) == steps
                got.append((a, b, c, wb))
            for x, y in zip(*got):
                assert np.array_equal(x, y), f"layer {li}: overlapped and serialised steps differ"
            th, m, v = th0[li].copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
            wb = np.zeros(n, np.uint16)
            for t in range(1, steps + 1):
                oracle.layer_step([pu.unit_grad_host(w, li, t, r) for r in range(R)], th, m, v, wb, hp_or, t)
            pu.assert_parity([pu.compare_fp32(f"theta l{li}", got[0][0], th),
                              pu.compare_fp32(f"m l{li}", got[0][1], m),
                              pu.compare_fp32(f"v l{li}", got[0][2], v),
                              pu.compare_bf16(f"w l{li}", got[0][3], wb)])
    finally:
        S.slide_state_destroy(overlapped)
        S.slide_state_destroy(serialised)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("clip", [0.0, 1e-3])
@pytest.mark.parametrize("fp32", [False, True])
def test_small_parity_with_finite_check(S, R, clip, fp32):
    """The kernels with the non-finite check compiled in: on finite inputs the
    same results as the oracle (bit for bit without the clip) and no flag."""
    reps = run_small(S, [9, 4096 + 3, (1 << 20) + 5], R, clip=clip, steps=3, fp32=fp32,
                     flags=S.SLIDE_FLAG_CHECK_FINITE)
    if clip == 0.0:
        for r in reps:
            assert r["not_bit_equal"] == 0, r


def test_external_bf16_out_and_empty_layer(S):
    run_small(S, [0, 5, 4099], 2, clip=0.5, bf16_external=True)


def test_prewarm_handoff_from_oracle(S):
    """m and v from 5 oracle steps handed to the state (t = 5), then GPU steps
    6..9 compared with oracle steps 6..9."""
    n, R = 70001, 4
    w = W.Workload("prewarm", [W.Unit("l", [("flat", n)])], R=R, steps=4, seed=21, max_grad_norm=1.0,
                   prewarm_steps=5)
    hp_or = pu.hp_oracle(w)
    th = synth.master(n, w.seed)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 6):
        oracle.layer_step([pu.unit_grad_host(w, 0, t, r) for r in range(R)], th, m, v, None, hp_or, t)
    st = S.slide_state_create([n], R)
    try:
        S.slide_layer_set(st, 0, th, m, v, step=5)
        grads = [dev_u16(n) for _ in range(R)]
        hp = S.hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_grad_norm)
        wb = np.zeros(n, np.uint16)
        for t in range(6, 10):
            for r in range(R):
                pu.unit_grad_dev(w, 0, t, r, grads[r].data_ptr())
            S.slide_layer_step(st, 0, grads, hp)
            oracle.layer_step([pu.unit_grad_host(w, 0, t, r) for r in range(R)], th, m, v, wb, hp_or, t)
        gt, gm, gv = (np.empty(n, np.float32) for _ in range(3))
        gw = np.empty(n, np.uint16)
        assert S.slide_layer_get(st, 0, gt, gm, gv, gw) == 9
        pu.assert_parity([pu.compare_fp32("theta", gt, th), pu.compare_fp32("m", gm, m),
                          pu.compare_fp32("v", gv, v), pu.compare_bf16("w", gw, wb)])
    finally:
        S.slide_state_destroy(st)


def test_write_set_is_exactly_the_layer(S):
    """A step of layer 0 touches exactly its own n elements: the next layer's
    arrays and an external output's bytes past n keep their sentinel values."""
    n0, n1, R = 4103, 333, 3
    st = S.slide_state_create([n0, n1], R)
    try:
        sent = np.full(n1, np.nan, np.float32)
        S.slide_layer_set(st, 1, sent, sent, sent, step=0)
        w = W.Workload("ws", [W.Unit("a", [("f", n0)])], R=R, steps=1, seed=3)
        grads = [dev_u16(n0) for _ in range(R)]
        for r in range(R):
            pu.unit_grad_dev(w, 0, 1, r, grads[r].data_ptr())
        out = torch.full((n0 + 64,), 0x7ABC, dtype=torch.int16, device="cuda")
        S.slide_layer_step(st, 0, grads, S.hparams(), None, out)
        torch.cuda.synchronize()
        tail = out[n0:].cpu().numpy()
        assert np.all(tail == 0x7ABC)
        a, b, c = (np.empty(n1, np.float32) for _ in range(3))
        S.slide_layer_get(st, 1, a, b, c)
        assert np.isnan(a).all() and np.isnan(b).all() and np.isnan(c).all()
    finally:
        S.slide_state_destroy(st)


def test_nonfinite_flag_reports_without_fault(S):
    n, R = 1000, 2
    st = S.slide_state_create([n], R, flags=S.SLIDE_FLAG_CHECK_FINITE)
    try:
        g = [torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        S.slide_layer_step(st, 0, g, S.hparams())
        assert S.slide_layer_status(st, 0) == S.SLIDE_OK
        g[1][17] = float("nan")
        S.slide_layer_step(st, 0, g, S.hparams())
        assert S.slide_layer_status(st, 0) == S.SLIDE_ERR_NONFINITE
        assert S.slide_layer_status(st, 0) == S.SLIDE_OK  # the mark is cleared
    finally:
        S.slide_state_destroy(st)


def test_argument_errors(S):
    n, R = 100, 2
    st = S.slide_state_create([n], R)
    try:
        g = [torch.zeros(n + 16, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        with pytest.raises(S.SlideError) as e:
            S.slide_layer_step(st, 0, [g[0], g[1].data_ptr() + 2], S.hparams())
        assert e.value.status == S.SLIDE_ERR_INVALID_ARG
        with pytest.raises(S.SlideError) as e:
            S.slide_layer_step(st, 1, g, S.hparams())
        assert e.value.status == S.SLIDE_ERR_INVALID_ARG
        with pytest.raises(S.SlideError) as e:
            S.slide_layer_step(st, 0, g, S.hparams(beta1=1.0))
        assert e.value.status == S.SLIDE_ERR_INVALID_ARG
        with pytest.raises(S.SlideError) as e:
            S.slide_model_step_streamed(st, 1, None, S.hparams())
        assert e.value.status == S.SLIDE_ERR_STATE
        # nothing was enqueued and t did not move
        assert S.slide_layer_get(st, 0) == 0
    finally:
        S.slide_state_destroy(st)


def test_state_allocation_matches_accounting(S):
    """cudaMemGetInfo sees the arena that slide_state_bytes predicts."""
    sizes = [100_000_000, 1]
    dev_bytes, host_bytes = S.slide_state_bytes(sizes, 4)
    assert host_bytes == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    st = S.slide_state_create(sizes, 4)
    try:
        free1, _ = torch.cuda.mem_get_info()
        used = free0 - free1
        assert dev_bytes <= used <= dev_bytes + (64 << 20), (used, dev_bytes)
    finally:
        S.slide_state_destroy(st)


# ---------------------------------------- full-size workloads, every element ----

def run_full_size(S, w):
    """The workload's single HBM-resident unit at full size, in the launch
    configuration the benchmark times (the library picks it), against the
    oracle run over the whole unit on the same seeded inputs: every element
    of master, m, v and the BF16 copy after the last step, and the clip
    coefficient of every step."""
    assert len(w.units) == 1
    n = w.units[0].numel
    hp_or = pu.hp_oracle(w)
    th = pu.master_threaded(n, w.seed)
    m, v, wb = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    grads = [dev_grad_buf(n, w.fp32_grads) for _ in range(w.R)]
    st = S.slide_state_create([n], w.R, flags=S.SLIDE_FLAG_FP32_GRADS if w.fp32_grads else 0)
    try:
        t0 = 0
        if w.prewarm_steps:
            # pre-warm m and v by the oracle over the whole unit, handed to the state
            for t in range(1, w.prewarm_steps + 1):
                for r in range(w.R):
                    pu.unit_grad_dev(w, 0, t, r, grads[r].data_ptr())
                reps = pu.replicas_to_host(w, 0, t, grads, n)
                pu.oracle_step_threaded(reps, th, m, v, None, hp_or, t)
                del reps
            S.slide_layer_set(st, 0, th, m, v, step=w.prewarm_steps)
            t0 = w.prewarm_steps
        else:
            synth.dev_master(S.slide_layer_ptrs(st, 0)[0], n, w.seed)   # the device twin of the same master
        hp = S.hparams(*w.hparams_tuple())
        for t in range(t0 + 1, t0 + w.steps + 1):
            for r in range(w.R):
                pu.unit_grad_dev(w, 0, t, r, grads[r].data_ptr())
            S.slide_layer_step(st, 0, grads, hp)
            reps = pu.replicas_to_host(w, 0, t, grads, n)
            coef = pu.oracle_step_threaded(reps, th, m, v, wb, hp_or, t)
            del reps
            if w.max_grad_norm > 0:
                gc = S.slide_layer_last_clip_coef(st, 0)
                assert abs(gc - coef) <= 2 * np.spacing(np.float32(coef)), (t, gc, coef)
        th_g, m_g, v_g = (np.empty(n, np.float32) for _ in range(3))
        w_g = np.empty(n, np.uint16)
        assert S.slide_layer_get(st, 0, th_g, m_g, v_g, w_g) == t0 + w.steps
        rep = [pu.compare_fp32_all("theta", th_g, th), pu.compare_fp32_all("m", m_g, m),
               pu.compare_fp32_all("v", v_g, v), pu.compare_bf16_all("w", w_g, wb)]
        pu.assert_parity(rep)
        assert np.array_equal(w_g, oracle.f32_to_bf16(th_g))
        if w.max_grad_norm <= 0:   # same FP32 operations on both sides without the clip
            assert all(r["not_bit_equal"] == 0 for r in rep), rep
        return rep
    finally:
        S.slide_state_destroy(st)


@pytest.mark.parametrize("name", ["h2560_R1", "h2560_R4_clip", "h5120_R8_logscale", "h2560_R4_clip_fp32grads"])
def test_full_size_workload_every_element(S, name):
    w = W.ALL[name]()
    rep = run_full_size(S, w)
    print(rep)
