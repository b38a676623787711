"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes the oracle against a closed form, a hand-derived exact
example, a library routine that implements the same textbook definition, or a
brute force, so that a plausible slip in the oracle (a dropped term, a wrong
sign or index, swapped betas, a misplaced eps, a wrong step count in the bias
correction, summing instead of averaging the replicas) fails at least one of
them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_exact(vals):
    """BF16 bit patterns of values that are exactly representable in BF16."""
    x = np.asarray(vals, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def random_bf16(rng, n, scale):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    return oracle.f32_to_bf16(x)


def ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(np.maximum(x, np.float32(1e-38))).astype(np.float64)


# ---------------------------------------------------------------- BF16 ----

def test_bf16_rounding_fixed_patterns():
    cases = {
        0x3F800000: 0x3F80,  # 1.0
        0x3F808000: 0x3F80,  # exact tie, kept bit even -> down
        0x3F818000: 0x3F82,  # exact tie, kept bit odd -> up
        0x3F808001: 0x3F81,  # just above the tie -> up
        0x3F807FFF: 0x3F80,  # just below the tie -> down
        0xBF818000: 0xBF82,  # negative tie to even
        0x7F7FFFFF: 0x7F80,  # largest finite float rounds to +inf
        0xFF7FFFFF: 0xFF80,
        0x7F800000: 0x7F80,  # +inf stays
        0x00000001: 0x0000,  # smallest subnormal rounds to zero
        0x00008000: 0x0000,  # subnormal tie to even (zero)
        0x00018000: 0x0002,  # subnormal tie to even (up)
        0x80000000: 0x8000,  # -0
    }
    for bits, want in cases.items():
        x = np.array([bits], np.uint32).view(np.float32)[0]
        assert oracle.lib().oracle_f32_to_bf16_rne(x) == want, hex(bits)
    # NaNs stay NaNs (the quiet bit is set so a payload cannot turn into inf)
    for bits in (0x7F800001, 0x7FC00000, 0xFF800001):
        x = np.array([bits], np.uint32).view(np.float32)[0]
        h = oracle.lib().oracle_f32_to_bf16_rne(x)
        assert (h & 0x7F80) == 0x7F80 and (h & 0x7F) != 0
        assert (h >> 15) == (bits >> 31)


def test_bf16_rounding_matches_torch():
    """torch's CPU float -> bfloat16 conversion is round-to-nearest-even."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # add ties and near-ties around random values
    ties = (bits & 0xFFFF0000) | 0x8000
    allb = np.concatenate([bits, ties, ties + 1, ties - 1]).astype(np.uint32)
    x = allb.view(np.float32)
    finite = np.isfinite(x)
    x = x[finite]
    ours = oracle.f32_to_bf16(x)
    theirs = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    back = oracle.bf16_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(theirs.view(np.int16).copy())
                          .view(torch.bfloat16).float().numpy())


# ------------------------------------------------------ closed forms ----

def test_step1_from_zero_moments_closed_form():
    """t = 1, m = v = 0: m_hat = g, v_hat = g^2, so
    theta1 = theta0*(1 - lr*wd) - lr*g/(|g| + eps), for every |g| including the
    eps regime (|g| ~ eps), where a misplaced eps would show."""
    rng = np.random.default_rng(1)
    n = 6000
    mags = np.concatenate([
        rng.standard_normal(2000) * 1e-3,
        rng.standard_normal(2000) * 1e-8,      # ~eps
        rng.standard_normal(2000) * 1e-10,     # << eps
    ])
    g = oracle.f32_to_bf16(mags.astype(np.float32))
    gv = oracle.bf16_to_f32(g).astype(np.float64)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    w = np.zeros(n, np.uint16)
    lr, wd, eps = 1e-5, 0.01, 1e-8
    hp = oracle.hparams(lr=lr, weight_decay=wd, eps=eps)
    oracle.layer_step([g], theta, m, v, w, hp, 1)
    lr64, wd64, eps64 = (float(np.float32(a)) for a in (lr, wd, eps))
    want = theta0.astype(np.float64) * (1 - lr64 * wd64) - lr64 * gv / (np.abs(gv) + eps64)
    err = np.abs(theta.astype(np.float64) - want)
    # rounding of theta itself plus a few FP32 roundings of the lr-sized term
    assert np.all(err <= 3 * ulp32(want) + lr64 * 2.0 ** -21), err.max()
    # and the moments are the textbook first step
    assert np.allclose(m, (1 - np.float32(0.9)) * gv, rtol=1e-6, atol=0)
    assert np.allclose(v, (1 - np.float32(0.999)) * gv * gv, rtol=1e-6, atol=0)


def test_zero_gradient_zero_state_is_pure_decay():
    """g = 0, m = v = 0: the Adam term is 0/eps = 0, so each step is exactly
    one FP32 multiply by (1 - lr*wd) and the moments stay exactly 0."""
    rng = np.random.default_rng(2)
    n = 1000
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    zero = np.zeros(n, np.uint16)
    hp = oracle.hparams()
    decay = np.float32(1.0 - float(np.float32(1e-5)) * float(np.float32(0.01)))
    want = theta0.copy()
    for t in range(1, 6):
        oracle.layer_step([zero, zero], theta, m, v, None, hp, t)
        want = (want * decay).astype(np.float32)
        assert np.array_equal(theta, want)
        assert not m.any() and not v.any()


@pytest.mark.parametrize("R", [2, 4, 8])
def test_identical_replicas_equal_one_replica(R):
    """The sum of R identical BF16 values is exact in FP32 for R <= 8 and R is a
    power of two, so the mean of R identical replicas is bit-identical to one."""
    rng = np.random.default_rng(3 + R)
    n = 3001
    g = random_bf16(rng, n, 1e-3)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = oracle.hparams(max_grad_norm=0.0)
    outs = []
    for reps in (1, R):
        theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        w = np.zeros(n, np.uint16)
        for t in range(1, 4):
            oracle.layer_step([g] * reps, theta, m, v, w, hp, t)
        outs.append((theta, m, v, w))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_replica_mean_is_elementwise_mean():
    """Replicas with different per-element values: the mean uses replica r's
    element i (not a shifted index, not the sum), exact here because the values
    are small integers times powers of two."""
    rng = np.random.default_rng(5)
    n = 257
    ks = rng.integers(-20, -4, size=n)
    reps = []
    for r in range(3):
        ints = rng.integers(-8, 9, size=n)
        reps.append(bf16_exact((ints * np.exp2(ks)).astype(np.float32)))
    gm = oracle.grad_mean(reps)
    exact = sum(oracle.bf16_to_f32(g).astype(np.float64) for g in reps) / 3.0
    # the sum is exact in FP32; one rounding of the division by 3
    assert np.all(np.abs(gm - exact) <= 0.5 * ulp32(exact) + 0)
    gm2 = oracle.grad_mean(reps[:2])
    exact2 = (oracle.bf16_to_f32(reps[0]).astype(np.float64)
              + oracle.bf16_to_f32(reps[1])) / 2.0
    assert np.array_equal(gm2.astype(np.float64), exact2)


def test_sign_sgd_limit_beta_zero():
    """beta1 = beta2 = 0, wd = 0: bc1 = bc2 = 1, m = g, v = g^2 at every step,
    so theta_t = theta_{t-1} - lr*g_t/(|g_t| + eps) for every t."""
    rng = np.random.default_rng(6)
    n = 2000
    theta = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    hp = oracle.hparams(beta1=0.0, beta2=0.0, weight_decay=0.0, lr=1e-3, eps=1e-8)
    lr64, eps64 = float(np.float32(1e-3)), float(np.float32(1e-8))
    for t in range(1, 5):
        g = random_bf16(rng, n, 10.0 ** rng.uniform(-9, -2))
        gv = oracle.bf16_to_f32(g).astype(np.float64)
        prev = theta.astype(np.float64)
        oracle.layer_step([g], theta, m, v, None, hp, t)
        want = prev - lr64 * gv / (np.abs(gv) + eps64)
        assert np.all(np.abs(theta - want) <= 3 * ulp32(want) + lr64 * 2.0 ** -21)


def test_constant_gradient_bias_correction_every_step():
    """A constant gradient g with wd = 0: m_t = g(1 - b1^t), v_t = g^2(1 - b2^t),
    so the bias-corrected moments are exactly g and g^2 at every t and each
    step moves theta by -lr*g/(|g| + eps).  A wrong t (t-1, t+1, a global
    count) or a dropped correction breaks this at small t."""
    rng = np.random.default_rng(8)
    n = 512
    g = random_bf16(rng, n, 1e-3)
    gv = oracle.bf16_to_f32(g).astype(np.float64)
    theta = np.zeros(n, np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    lr = 1e-2
    hp = oracle.hparams(lr=lr, weight_decay=0.0)
    lr64, eps64 = float(np.float32(lr)), float(np.float32(1e-8))
    step = -lr64 * gv / (np.abs(gv) + eps64)
    for t in range(1, 41):
        prev = theta.astype(np.float64)
        oracle.layer_step([g], theta, m, v, None, hp, t)
        d = theta.astype(np.float64) - prev
        assert np.allclose(d, step, rtol=2e-5, atol=2 * ulp32(theta).max()), t


def _load_golden(name):
    rows, params = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) == 2:
                params[parts[0]] = Fraction(parts[1])
            else:
                rows.append([int(parts[0])] + [Fraction(p) for p in parts[1:]])
    return params, rows


def test_hand_worked_three_steps():
    p, rows = _load_golden("adamw_three_step_exact.txt")
    hp = oracle.hparams(lr=float(p["lr"]), beta1=float(p["beta1"]), beta2=float(p["beta2"]),
                        eps=float(p["eps"]), weight_decay=float(p["weight_decay"]))
    theta = np.array([float(p["theta0"])], np.float32)
    m, v = np.zeros(1, np.float32), np.zeros(1, np.float32)
    th64, m64, v64 = (np.array([float(p["theta0"])]), np.zeros(1), np.zeros(1))
    for step, grad, m_want, v_want, th_rat, th_c, th_arg in rows:
        g = bf16_exact([float(grad)])
        oracle.layer_step([g], theta, m, v, None, hp, step)
        oracle.layer_step_f64([g], th64, m64, v64, hp, step)
        th_want = float(th_rat) + float(th_c) * float(th_arg) ** 0.5
        assert m[0] == float(m_want) and v[0] == float(v_want), step
        assert abs(theta[0] - th_want) <= 2e-7 * abs(th_want), (step, theta[0], th_want)
        assert abs(th64[0] - th_want) <= 1e-15 * abs(th_want)
        assert m64[0] == float(m_want) and v64[0] == float(v_want)


# ---------------------------------------------------------------- clip ----

def test_clip_hand_built():
    """Two replicas [1,0,1,0] and [0,1,0,1]: the mean is [1/2]*4, whose L2 norm
    is exactly 1 (the sum would have norm 2).  With c = 1/2 the norm is 2c and
    coef = c/(2c + 1e-6); with c = 2 nothing is clipped.  The clipped gradient
    is what enters the first moment: m1 = (1 - b1)*coef*g."""
    a = bf16_exact([1, 0, 1, 0])
    b = bf16_exact([0, 1, 0, 1])
    gm = oracle.grad_mean([a, b])
    assert np.array_equal(gm, np.full(4, 0.5, np.float32))
    assert oracle.grad_sqnorm(gm) == 1.0
    coef = oracle.clip_coef(1.0, 0.5)
    assert coef == np.float32(0.5 / (1.0 + 1e-6))
    assert oracle.clip_coef(1.0, 2.0) == 1.0
    assert oracle.clip_coef(1.0, 0.0) == 1.0  # clip off
    for c, k in ((0.5, coef), (2.0, 1.0)):
        theta, m, v = np.zeros(4, np.float32), np.zeros(4, np.float32), np.zeros(4, np.float32)
        got = oracle.layer_step([a, b], theta, m, v, None, oracle.hparams(max_grad_norm=c), 1)
        assert got == np.float32(k)
        g = np.float32(0.5) * np.float32(k)
        assert np.all(m == np.float32(1 - np.float32(0.9)) * g)


# --------------------------------------------- library routine: torch ----

@pytest.mark.parametrize("gdt", ["bf16", "f32"])
@pytest.mark.parametrize("R,clip", [(1, 0.0), (3, 0.0), (4, 1.0), (8, 1e-3)])
def test_matches_torch_adamw_float64(R, clip, gdt):
    """torch.optim.AdamW (decoupled decay, bias correction, eps after the square
    root of the corrected second moment) and torch.nn.utils.clip_grad_norm_
    (coef = c/(norm + 1e-6), clamped at 1), run in float64 on the mean of the
    same BF16 replicas, are the textbook step this oracle reads the pages as.
    FP32 oracle within 2e-6*(1+|x|) on theta, m, v; the float64 brute force
    within 1e-12 relative."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(100 + R)
    n = 4096
    lr, b1, b2, eps, wd = (float(np.float32(x)) for x in (1e-3, 0.9, 0.999, 1e-8, 0.01))
    hp = oracle.hparams(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd, max_grad_norm=clip)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    th64, m64, v64 = theta0.astype(np.float64), np.zeros(n), np.zeros(n)
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    scales = 10.0 ** rng.uniform(-9, -2, size=n)
    for t in range(1, 21):
        raw = [(rng.standard_normal(n) * scales).astype(np.float32) for _ in range(R)]
        grads = raw if gdt == "f32" else [oracle.f32_to_bf16(x) for x in raw]
        oracle.layer_step(grads, theta, m, v, None, hp, t)
        oracle.layer_step_f64(grads, th64, m64, v64, hp, t)
        vals = raw if gdt == "f32" else [oracle.bf16_to_f32(g) for g in grads]
        mean = sum(x.astype(np.float64) for x in vals) / R
        p.grad = torch.from_numpy(mean)
        if clip > 0:
            torch.nn.utils.clip_grad_norm_([p], float(np.float32(clip)))
        opt.step()
        st = opt.state[p]
        tp, tm, tv = p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        assert np.all(np.abs(theta - tp) <= 2e-6 * (1 + np.abs(tp))), t
        assert np.all(np.abs(m - tm) <= 2e-6 * (1 + np.abs(tm))), t
        assert np.all(np.abs(v - tv) <= 2e-6 * (1 + np.abs(tv))), t
        # sharper than the GPU tolerance: FP32 roundings relative to each
        # element's own gradient scale (m can cancel to ~0, hence the atol)
        assert np.allclose(m, tm, rtol=1e-5, atol=0) or np.all(
            np.abs(m - tm) <= 1e-5 * np.abs(tm) + 1e-6 * scales)
        assert np.all(np.abs(v - tv) <= 1e-5 * np.abs(tv) + 1e-6 * scales ** 2)
        assert np.allclose(th64, tp, rtol=1e-12, atol=1e-18)
        assert np.all(np.abs(m64 - tm) <= 1e-12 * np.abs(tm) + 1e-14 * scales)
        assert np.all(np.abs(v64 - tv) <= 1e-12 * np.abs(tv) + 1e-14 * scales ** 2)


# ---------------------------------------------- float64 brute force ----

@pytest.mark.parametrize("R,clip", [(1, 0.0), (4, 1.0), (8, 0.0)])
def test_fp32_oracle_vs_float64_brute_force(R, clip):
    """1k elements, the workloads' hyper-parameters, 20 steps: the FP32 oracle
    stays within 1e-6*(1+|x|) of the float64 brute force on theta, and its
    emitted BF16 is the RNE rounding of its own FP32 master, bit for bit."""
    rng = np.random.default_rng(200 + R)
    n = 1000
    hp = oracle.hparams(max_grad_norm=clip)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    w = np.zeros(n, np.uint16)
    th64, m64, v64 = theta0.astype(np.float64), np.zeros(n), np.zeros(n)
    sig = 10.0 ** rng.uniform(-5, -2, size=n)
    for t in range(1, 21):
        grads = [oracle.f32_to_bf16((rng.standard_normal(n) * sig).astype(np.float32))
                 for _ in range(R)]
        c32 = oracle.layer_step(grads, theta, m, v, w, hp, t)
        c64 = oracle.layer_step_f64(grads, th64, m64, v64, hp, t)
        assert abs(c32 - c64) <= 1e-7 * c64
        assert np.all(np.abs(theta - th64) <= 1e-6 * (1 + np.abs(th64)))
        assert np.all(np.abs(m - m64) <= 1e-6 * (1 + np.abs(m64)))
        assert np.all(np.abs(v - v64) <= 1e-6 * (1 + np.abs(v64)))
        assert np.array_equal(w, oracle.f32_to_bf16(theta))


def test_step_scalars():
    """The per-step scalars are the bias corrections of step t (not t-1)."""
    hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.999, weight_decay=0.1)
    for t in (1, 2, 10, 1000):
        s = oracle.step_scalars(hp, t)
        b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
        assert s.step_size == np.float32(float(np.float32(1e-3)) / (1 - b1 ** t))
        assert s.bc2_sqrt == np.float32((1 - b2 ** t) ** 0.5)
        assert s.decay == np.float32(1 - float(np.float32(1e-3)) * float(np.float32(0.1)))


def test_empty_layer():
    theta = np.zeros(0, np.float32)
    c = oracle.layer_step([np.zeros(0, np.uint16)], theta, theta.copy(), theta.copy(),
                          np.zeros(0, np.uint16), oracle.hparams(max_grad_norm=1.0), 1)
    assert c == 1.0


# ---------------------------------------------- FP32 gradient replicas ----

def test_f32_replica_mean_is_elementwise_mean():
    """FP32 replicas: replica r's element i enters the mean of element i, and
    the result is the sum divided by R (exact on these small dyadic values)."""
    rng = np.random.default_rng(55)
    n = 301
    k = rng.integers(-30, -10, size=n)            # one exponent per element, shared by the replicas
    reps = [(rng.integers(-1000, 1001, size=n) * np.exp2(k)).astype(np.float32) for _ in range(4)]
    gm = oracle.grad_mean(reps)
    exact = sum(x.astype(np.float64) for x in reps) / 4.0
    assert np.array_equal(gm.astype(np.float64), exact)
    gm3 = oracle.grad_mean(reps[:3])
    ex3 = sum(x.astype(np.float64) for x in reps[:3]) / 3.0
    assert np.all(np.abs(gm3 - ex3) <= 0.5 * ulp32(ex3))


def test_f32_identical_replicas_equal_one_replica():
    """Values with at most 20 significant bits: every partial sum of up to 8
    copies (at most 8x) fits in FP32's 24 bits, so the mean equals the single
    replica bit for bit."""
    rng = np.random.default_rng(56)
    n = 2049
    x = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    x = (x.view(np.uint32) & np.uint32(0xFFFFFFF8)).view(np.float32)   # 20 significant bits
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    outs = []
    for reps in (1, 2, 4, 8):
        th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        w = np.zeros(n, np.uint16)
        for t in range(1, 4):
            oracle.layer_step([x] * reps, th, m, v, w, oracle.hparams(), t)
        outs.append((th, m, v, w))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a, b)


def test_f32_step1_closed_form():
    rng = np.random.default_rng(57)
    n = 3000
    g = np.concatenate([rng.standard_normal(1000) * 1e-3, rng.standard_normal(1000) * 1e-8,
                        rng.standard_normal(1000) * 1e-11]).astype(np.float32)
    th0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.layer_step([g], th, m, v, None, oracle.hparams(), 1)
    lr64, wd64, eps64 = (float(np.float32(a)) for a in (1e-5, 0.01, 1e-8))
    gv = g.astype(np.float64)
    want = th0.astype(np.float64) * (1 - lr64 * wd64) - lr64 * gv / (np.abs(gv) + eps64)
    assert np.all(np.abs(th - want) <= 3 * ulp32(want) + lr64 * 2.0 ** -21)


@pytest.mark.parametrize("clip", [0.0, 1.0])
def test_openmp_build_is_the_same_oracle(clip):
    """The -fopenmp build (used only to time the oracle on all cores) splits
    the element loops across threads without changing any element's
    operations: without the clip it is bit-identical to the single-threaded
    build; with it, only the clip's double sum changes order, so the clip
    coefficients agree to within an FP32 ulp and the states to within what
    one ulp of the coefficient can move."""
    rng = np.random.default_rng(7)
    n, R = 300_001, 4
    grads = [oracle.f32_to_bf16(rng.standard_normal(n).astype(np.float32) * 1e-3) for _ in range(R)]
    th0 = rng.standard_normal(n).astype(np.float32) * 0.02
    hp = oracle.hparams(max_grad_norm=clip)
    runs = {}
    for omp in (False, True):
        th, m, v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        w = np.zeros(n, np.uint16)
        coefs = [oracle.layer_step(grads, th, m, v, w, hp, t, openmp=omp) for t in (1, 2)]
        runs[omp] = (coefs, th, m, v, w)
    assert oracle.threads(False) == 1
    assert oracle.threads(True) >= 1
    (c0, *state0), (c1, *state1) = runs[False], runs[True]
    if clip == 0.0:
        assert c0 == c1 == [1.0, 1.0]
        for a, b in zip(state0, state1):
            assert np.array_equal(a, b)
    else:
        for a, b in zip(c0, c1):
            assert abs(a - b) <= np.spacing(np.float32(a))
        assert np.allclose(state0[0], state1[0], rtol=0, atol=1e-9)
        assert np.allclose(state0[1], state1[1], rtol=2e-7, atol=0)
