"""GPU tests of the host-resident streamed step (slide_model_step_streamed).

A toy model of units of mixed sizes (including an empty one) runs with a tiny
copy chunk so the slot handoff between the copy-out of one unit and the
copy-in of the next happens over many chunks; every element is compared with
the oracle after each step.  The invariants of synchronous data parallelism
are checked: one update per unit per step (every t moves by exactly one),
same version on entry (SLIDE_ERR_VERSION otherwise), and a sweep that stops
part-way leaves the state marked until a common version is restored.
Failures are made on the host (a callback that returns an error, a wait
limit shorter than the work); no GPU fault, trap or hang is involved.
"""
import ctypes as C

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


class ModelGradsHolder:
    """synth.ModelGrads with its arrays kept alive."""

    def __init__(self, w: W.Workload, step: int):
        self.numel = (C.c_int64 * len(w.units))(*[u.numel for u in w.units])
        segs_b, offs, lens, scs = [0], [], [], []
        for ui, u in enumerate(w.units):
            for (off, n), sc in zip(u.segments(), w.tensor_scales(ui)):
                offs.append(off)
                lens.append(n)
                scs.append(sc)
            segs_b.append(len(offs))
        self.seg_begin = (C.c_int32 * len(segs_b))(*segs_b)
        self.seg_off = (C.c_int64 * len(offs))(*offs)
        self.seg_len = (C.c_int64 * len(lens))(*lens)
        self.seg_scale = (C.c_float * len(scs))(*scs)
        self.mg = synth.ModelGrads(synth.spec(w.seed, w.grad_kind, w.zero_prob), len(w.units), w.R, step, 0,
                                   C.cast(self.numel, C.c_void_p), C.cast(self.seg_begin, C.c_void_p),
                                   C.cast(self.seg_off, C.c_void_p), C.cast(self.seg_len, C.c_void_p),
                                   C.cast(self.seg_scale, C.c_void_p), w.grad_scale, int(w.fp32_grads))


def init_streamed(S, w, st):
    """Seeded master in the pinned host state (written by the GPU through the
    memory's device address), m = v = 0, BF16 copy = bf16(master)."""
    for ui, u in enumerate(w.units):
        th = synth.master(u.numel, w.seed, unit=ui)
        S.slide_layer_set(st, ui, master=th, step=0)


def check_timeline(S, st, sizes):
    """The engine's per-unit events of the last step respect causality: the
    master lands after its copy-in began and before the copy-in ends; the
    updates end after the copy-in ends; the write-back starts after the master
    landed (the first chunk's update needs it) and ends after the last update;
    units are written back in reverse order."""
    units, fwd_end = S.slide_streamed_timeline(st)
    assert np.isfinite(fwd_end) and fwd_end >= 0
    eps = 1e-3
    for u in units:
        assert all(np.isfinite(list(u.values()))), u
        assert u["h2d_begin"] <= u["master_landed"] + eps <= u["h2d_end"] + 2 * eps, u
        assert u["h2d_end"] <= u["update_end"] + eps, u
        assert u["master_landed"] <= u["d2h_begin"] + eps, u
        assert u["update_end"] <= u["d2h_end"] + eps and u["d2h_begin"] <= u["d2h_end"] + eps, u
    ends = [u["d2h_end"] for u in units]
    assert all(ends[l] >= ends[l + 1] - eps for l in range(len(units) - 1))
    # host enqueue order: a unit's copy-in is enqueued before its update, and
    # the units of the reverse sweep one after another
    for l, u in enumerate(units):
        assert u["host_copyin_enqueued"] <= u["host_unit_enqueued"], u
        if l + 1 < len(units):
            assert units[l + 1]["host_unit_enqueued"] <= u["host_unit_enqueued"], (l, u)


def toy(R=3, clip=0.0, seed=5, fp32=False):
    sizes = [5000, 70001, (1 << 20) + 3, 0, 777, 123457]
    return W.Workload("toy", [W.Unit(f"u{i}", [("a", n // 2), ("b", n - n // 2)]) for i, n in enumerate(sizes)],
                      R=R, steps=3, seed=seed, max_grad_norm=clip, lr=1e-3, streamed=True, fp32_grads=fp32)


def pinned_arena(nbytes):
    """Caller-owned pinned host memory of at least nbytes, 256-byte aligned:
    (keep-alive tensor, address)."""
    t = torch.empty(nbytes + 256, dtype=torch.uint8, pin_memory=True)
    addr = (t.data_ptr() + 255) // 256 * 256
    return t, addr


@pytest.mark.parametrize("clip,chunk,chunk_d2h,fp32,in_hbm,arena", [
    (0.0, 64 << 10, 0, False, False, False), (0.5, 256, 0, False, False, False),
    (1e4, 1 << 20, 0, False, False, False), (0.0, 64 << 10, 0, True, False, False),
    (0.5, 4096, 0, True, False, False), (0.0, 64 << 10, 0, False, True, False),
    (0.5, 4096, 0, True, True, False),
    # write-back chunks smaller, larger and not a multiple of the copy-in chunks
    (0.0, 64 << 10, 4096, False, False, False), (0.5, 4096, 64 << 10, False, False, True),
    (0.0, 1024, 3072, True, True, True), (0.0, 768, 1 << 20, False, True, False),
    (1e-3, 3072, 1024, False, False, True),
    # the pinned state in a huge-page mapping registered with cudaHostRegister
    (0.5, 64 << 10, 0, False, False, "huge"), (0.0, 4096, 64 << 10, False, True, "huge")])
def test_streamed_toy_every_element(S, clip, chunk, chunk_d2h, fp32, in_hbm, arena):
    w = toy(clip=clip, fp32=fp32)
    flags = (S.SLIDE_FLAG_FP32_GRADS if fp32 else 0) | (S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0)
    if arena == "huge":
        flags |= S.SLIDE_FLAG_HOST_HUGE_PAGES
        arena = False
    sizes = [u.numel for u in w.units]
    keep, addr, nbytes = None, None, 0
    if arena:
        nbytes = S.slide_state_bytes(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)[1]
        keep, addr = pinned_arena(nbytes)
        keep.fill_(0x5A)          # the state must zero what it uses
    st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED,
                              chunk_bytes=chunk, chunk_bytes_d2h=chunk_d2h, flags=flags,
                              host_arena=addr, host_arena_bytes=nbytes)
    try:
        if arena:
            assert S.slide_layer_ptrs(st, 0)[0] == addr
        init_streamed(S, w, st)
        ref = []
        for ui, u in enumerate(w.units):
            ref.append([synth.master(u.numel, w.seed, unit=ui), np.zeros(u.numel, np.float32),
                        np.zeros(u.numel, np.float32), np.zeros(u.numel, np.uint16)])
        hp = S.hparams(*w.hparams_tuple())
        hp_or = pu.hp_oracle(w)
        for t in range(1, w.steps + 1):
            holder = ModelGradsHolder(w, t)
            S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, hp)
            for ui, u in enumerate(w.units):
                reps = [pu.unit_grad_host(w, ui, t, r) for r in range(w.R)]
                oracle.layer_step(reps, *ref[ui], hp_or, t)
                a, b, c = (np.empty(u.numel, np.float32) for _ in range(3))
                wb = np.empty(u.numel, np.uint16)
                assert S.slide_layer_get(st, ui, a, b, c, wb) == t
                rep = [pu.compare_fp32("theta", a, ref[ui][0]), pu.compare_fp32("m", b, ref[ui][1]),
                       pu.compare_fp32("v", c, ref[ui][2]), pu.compare_bf16("w", wb, ref[ui][3])]
                pu.assert_parity(rep)
                # the host mirror that the next forward sweep delivers is bf16(master)
                assert np.array_equal(wb, oracle.f32_to_bf16(a))
                if clip == 0.0:
                    assert all(r["not_bit_equal"] == 0 for r in rep[:3]), rep
            check_timeline(S, st, [u.numel for u in w.units])
    finally:
        S.slide_state_destroy(st)


@pytest.mark.parametrize("in_hbm,chunk,chunk_d2h", [(False, 64 << 10, 0), (True, 4096, 64 << 10),
                                                   (False, 768, 1 << 20), (True, 1 << 20, 256)])
def test_streamed_async_steps_every_element(S, in_hbm, chunk, chunk_d2h):
    """Steps enqueued with slide_model_step_streamed_async back to back (each
    unit's next delivery and copy-in wait on the device for its own previous
    write-back), then mixed with a synchronous step and with accessors that
    must wait for a step in flight: every element against the oracle."""
    w = toy(clip=0.5)
    w.steps = 5
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0
    sizes = [u.numel for u in w.units]
    st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, chunk_bytes=chunk,
                              chunk_bytes_d2h=chunk_d2h, flags=flags)
    try:
        init_streamed(S, w, st)
        ref = [[synth.master(u.numel, w.seed, unit=ui), np.zeros(u.numel, np.float32),
                np.zeros(u.numel, np.float32), np.zeros(u.numel, np.uint16)] for ui, u in enumerate(w.units)]
        hp = S.hparams(*w.hparams_tuple())

        def compare(t):
            for ui, u in enumerate(w.units):
                a, b, c = (np.empty(u.numel, np.float32) for _ in range(3))
                wb = np.empty(u.numel, np.uint16)
                assert S.slide_layer_get(st, ui, a, b, c, wb) == t
                pu.assert_parity([pu.compare_fp32("theta", a, ref[ui][0]), pu.compare_fp32("m", b, ref[ui][1]),
                                  pu.compare_fp32("v", c, ref[ui][2]), pu.compare_bf16("w", wb, ref[ui][3])])

        def oracle_to(t0, t1):
            for t in range(t0, t1 + 1):
                for ui, u in enumerate(w.units):
                    oracle.layer_step([pu.unit_grad_host(w, ui, t, r) for r in range(w.R)], *ref[ui],
                                      pu.hp_oracle(w), t)

        # three asynchronous steps back to back, then a sync
        for t in (1, 2, 3):
            S.slide_model_step_streamed_async(st, synth.grad_fn_address(), ModelGradsHolder(w, t).mg, hp)
        S.slide_streamed_sync(st)
        oracle_to(1, 3)
        compare(3)
        # an asynchronous step read back without a sync (the accessor waits),
        # then a synchronous step behind another asynchronous one
        S.slide_model_step_streamed_async(st, synth.grad_fn_address(), ModelGradsHolder(w, 4).mg, hp)
        oracle_to(4, 4)
        compare(4)
        S.slide_model_step_streamed_async(st, synth.grad_fn_address(), ModelGradsHolder(w, 5).mg, hp)
        S.slide_model_step_streamed(st, synth.grad_fn_address(), ModelGradsHolder(w, 6).mg, hp)
        oracle_to(5, 6)
        compare(6)
        check_timeline(S, st, sizes)
        S.slide_streamed_sync(st)   # nothing pending: a no-op
    finally:
        S.slide_state_destroy(st)


@pytest.mark.parametrize("sizes,in_hbm", [([123_457], False), ([123_457], True), ([0, 70_001], False),
                                           ([70_001, 0], True), ([5, 3], False)])
def test_streamed_few_units_every_element(S, sizes, in_hbm):
    """Models of one or two units (one of them empty, or both tiny): the slot
    handoff with no neighbour, every element against the oracle for 3 steps."""
    w = W.Workload("few", [W.Unit(f"u{i}", [("a", n)]) for i, n in enumerate(sizes)], R=3, steps=3, seed=23,
                   max_grad_norm=0.5, lr=1e-3, streamed=True)
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if in_hbm else 0
    st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, chunk_bytes=4096, flags=flags)
    try:
        init_streamed(S, w, st)
        ref = [[synth.master(n, w.seed, unit=ui), np.zeros(n, np.float32), np.zeros(n, np.float32),
                np.zeros(n, np.uint16)] for ui, n in enumerate(sizes)]
        hp = S.hparams(*w.hparams_tuple())
        for t in range(1, w.steps + 1):
            holder = ModelGradsHolder(w, t)
            S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, hp)
            for ui, n in enumerate(sizes):
                oracle.layer_step([pu.unit_grad_host(w, ui, t, r) for r in range(w.R)], *ref[ui], pu.hp_oracle(w), t)
        for ui, n in enumerate(sizes):
            a, b, c = (np.empty(n, np.float32) for _ in range(3))
            wb = np.empty(n, np.uint16)
            assert S.slide_layer_get(st, ui, a, b, c, wb) == w.steps
            pu.assert_parity([pu.compare_fp32("theta", a, ref[ui][0]), pu.compare_fp32("m", b, ref[ui][1]),
                              pu.compare_fp32("v", c, ref[ui][2]), pu.compare_bf16("w", wb, ref[ui][3])])
    finally:
        S.slide_state_destroy(st)


def test_streamed_caller_arena_reused_by_states(S):
    """One caller-owned pinned arena serves two states in turn: the first
    state's steps leave it dirty, the second starts from zero state (the
    state zeroes what it uses), steps against the oracle, and destroying a
    state leaves the arena to its owner."""
    w1 = toy(R=2, seed=8)
    w2 = W.Workload("toy2", [W.Unit("a", [("a", 300_001)]), W.Unit("b", [("b", 65_537)])], R=4, steps=2, seed=9,
                    lr=1e-3, streamed=True)
    need = max(S.slide_state_bytes([u.numel for u in w.units], w.R,
                                   residency=S.SLIDE_RESIDENCY_HOST_STREAMED)[1] for w in (w1, w2))
    keep, addr = pinned_arena(need)
    for w in (w1, w2):
        sizes = [u.numel for u in w.units]
        st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, chunk_bytes=8192,
                                  host_arena=addr, host_arena_bytes=need)
        try:
            for ui, u in enumerate(w.units):
                m = np.empty(u.numel, np.float32)
                S.slide_layer_get(st, ui, m=m)
                assert not m.any()
            init_streamed(S, w, st)
            ref = [[synth.master(u.numel, w.seed, unit=ui), np.zeros(u.numel, np.float32),
                    np.zeros(u.numel, np.float32), np.zeros(u.numel, np.uint16)] for ui, u in enumerate(w.units)]
            hp = S.hparams(*w.hparams_tuple())
            for t in range(1, w.steps + 1):
                holder = ModelGradsHolder(w, t)
                S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, hp)
                for ui, u in enumerate(w.units):
                    oracle.layer_step([pu.unit_grad_host(w, ui, t, r) for r in range(w.R)], *ref[ui],
                                      pu.hp_oracle(w), t)
            for ui, u in enumerate(w.units):
                a, b, c = (np.empty(u.numel, np.float32) for _ in range(3))
                wb = np.empty(u.numel, np.uint16)
                S.slide_layer_get(st, ui, a, b, c, wb)
                rep = [pu.compare_fp32("theta", a, ref[ui][0]), pu.compare_fp32("m", b, ref[ui][1]),
                       pu.compare_fp32("v", c, ref[ui][2]), pu.compare_bf16("w", wb, ref[ui][3])]
                pu.assert_parity(rep)
                assert all(r["not_bit_equal"] == 0 for r in rep), rep
        finally:
            S.slide_state_destroy(st)
    keep.fill_(1)                       # still the caller's memory
    assert int(keep[addr - keep.data_ptr()]) == 1


def test_streamed_caller_arena_rejected(S):
    sizes = [10_000]
    need = S.slide_state_bytes(sizes, 1, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)[1]
    keep, addr = pinned_arena(need)
    with pytest.raises(S.SlideError) as e:
        S.slide_state_create(sizes, 1, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, host_arena=addr,
                             host_arena_bytes=need - 256)
    assert e.value.status == S.SLIDE_ERR_INVALID_ARG and "smaller" in str(e.value)
    pageable = np.zeros(need + 256, np.uint8)
    paddr = (pageable.ctypes.data + 255) // 256 * 256
    with pytest.raises(S.SlideError) as e:
        S.slide_state_create(sizes, 1, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, host_arena=paddr,
                             host_arena_bytes=need)
    assert e.value.status == S.SLIDE_ERR_INVALID_ARG and "pinned" in str(e.value)


def test_streamed_python_callback_sees_master_and_errors_abort(S):
    """A Python callback (ctypes) receives R writable replica buffers plus the
    unit's FP32 master in the window; returning non-zero at one unit aborts
    the sweep: units already written back carry the new version, the rest the
    old one, and the state refuses further steps until restored."""
    sizes = [1000, 2000, 3000, 4000]
    R = 2
    st = S.slide_state_create(sizes, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, chunk_bytes=4096)
    seen = []

    def cb(user, layer, ptrs, stream):
        n = sizes[layer]
        seen.append((layer, ptrs[R] is not None))
        for r in range(R):  # zero gradients: the generator with scale 0
            synth.dev_grad(ptrs[r], n, synth.spec(1), layer, 1, r, 0.0, stream=stream or 0)
        return 7 if (fail_at[0] is not None and layer == fail_at[0]) else 0

    fail_at = [None]
    fn = S.SLIDE_GRAD_FN(cb)
    try:
        for ui, n in enumerate(sizes):
            S.slide_layer_set(st, ui, master=np.full(n, 0.5, np.float32), step=0)
        S.slide_model_step_streamed(st, fn, None, S.hparams())
        assert [l for l, _ in seen] == [3, 2, 1, 0] and all(has for _, has in seen)
        assert [S.slide_layer_get(st, i) for i in range(4)] == [1, 1, 1, 1]
        fail_at[0] = 1
        with pytest.raises(S.SlideError) as e:
            S.slide_model_step_streamed(st, fn, None, S.hparams())
        assert e.value.status == S.SLIDE_ERR_ABORTED
        # reverse sweep order 3, 2, 1: units 3 and 2 were updated, 1 and 0 not
        assert [S.slide_layer_get(st, i) for i in range(4)] == [1, 1, 2, 2]
        fail_at[0] = None
        with pytest.raises(S.SlideError) as e:
            S.slide_model_step_streamed(st, fn, None, S.hparams())
        assert e.value.status == S.SLIDE_ERR_ABORTED
        for ui, n in enumerate(sizes):
            S.slide_layer_set(st, ui, master=np.full(n, 0.5, np.float32), step=4)
        S.slide_model_step_streamed(st, fn, None, S.hparams())
        assert [S.slide_layer_get(st, i) for i in range(4)] == [5, 5, 5, 5]
    finally:
        S.slide_state_destroy(st)


def test_streamed_callback_gets_resident_bf16_copy(S):
    """With the BF16 copy kept in HBM the callback is handed each unit's
    resident BF16 compute copy (what a backward pass reads there), holding
    bf16 of the master before this step's update."""
    sizes = [3000, 70001, 5000]
    R = 2
    st = S.slide_state_create(sizes, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, chunk_bytes=8192,
                              flags=S.SLIDE_FLAG_BF16_COPY_IN_HBM)
    seen = {}
    snaps = {ui: torch.empty(n, dtype=torch.int16, device="cuda") for ui, n in enumerate(sizes)}

    class DevView:
        def __init__(self, ptr, n):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i2", "data": (ptr, False), "version": 2}

    def cb(user, layer, ptrs, stream):
        n = sizes[layer]
        seen[layer] = ptrs[R]
        # snapshot the weights handed over, on the callback's stream (before the update)
        with torch.cuda.stream(torch.cuda.ExternalStream(stream)):
            snaps[layer].copy_(torch.as_tensor(DevView(ptrs[R], n), device="cuda"))
        for r in range(R):
            synth.dev_grad(ptrs[r], n, synth.spec(1), layer, 1, r, 1e-3, stream=stream or 0)
        return 0

    fn = S.SLIDE_GRAD_FN(cb)
    try:
        masters = [synth.master(n, 4, unit=ui) for ui, n in enumerate(sizes)]
        for ui in range(len(sizes)):
            S.slide_layer_set(st, ui, master=masters[ui], step=0)
        S.slide_model_step_streamed(st, fn, None, S.hparams())
        assert sorted(seen) == [0, 1, 2]
        for ui in seen:
            assert seen[ui] == S.slide_layer_ptrs(st, ui)[3]
            # the callback saw bf16 of the master before the update
            assert np.array_equal(snaps[ui].cpu().numpy().view(np.uint16), oracle.f32_to_bf16(masters[ui]))
        # after the step the resident copy is bf16 of the new master
        for ui, n in enumerate(sizes):
            th = np.empty(n, np.float32)
            wb = np.empty(n, np.uint16)
            S.slide_layer_get(st, ui, master=th, bf16=wb)
            assert np.array_equal(wb, oracle.f32_to_bf16(th))
            assert not np.array_equal(th, masters[ui])
    finally:
        S.slide_state_destroy(st)


def test_streamed_version_gate(S):
    sizes = [100, 200]
    st = S.slide_state_create(sizes, 1, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    try:
        S.slide_layer_set(st, 1, step=3)
        w = W.Workload("v", [W.Unit("a", [("a", 100)]), W.Unit("b", [("b", 200)])], R=1, steps=1, seed=1)
        holder = ModelGradsHolder(w, 1)
        with pytest.raises(S.SlideError) as e:
            S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, S.hparams())
        assert e.value.status == S.SLIDE_ERR_VERSION
        # slide_layer_step is for the HBM residency only
        g = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(S.SlideError) as e:
            S.slide_layer_step(st, 0, [g], S.hparams())
        assert e.value.status == S.SLIDE_ERR_STATE
    finally:
        S.slide_state_destroy(st)


def test_streamed_wait_limit_returns_timeout(S):
    """A wait limit (1 ms) far shorter than the sweep: the host wait gives up
    with SLIDE_ERR_TIMEOUT while the GPU finishes normally; destroy then
    waits for the streams and the context stays usable."""
    sizes = [64 << 20, 64 << 20]
    R = 4
    st = S.slide_state_create(sizes, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, timeout_ms=1)
    try:
        w = W.Workload("to", [W.Unit("a", [("a", sizes[0])]), W.Unit("b", [("b", sizes[1])])], R=R, steps=1,
                       seed=2)
        holder = ModelGradsHolder(w, 1)
        with pytest.raises(S.SlideError) as e:
            S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, S.hparams())
        assert e.value.status == S.SLIDE_ERR_TIMEOUT
    finally:
        S.slide_state_destroy(st)
    x = torch.ones(1000, device="cuda")
    assert float(x.sum()) == 1000.0


def test_streamed_accounting_matches_allocation(S):
    """Pinned host bytes = master+m+v+BF16 copy of every unit (14 B/param plus
    256-byte alignment); the HBM window depends only on the largest unit."""
    sizes = [3_000_000, 5_000_000, 1_000]
    R = 4
    dev_b, host_b = S.slide_state_bytes(sizes, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    N = sum(sizes)
    assert 14 * N <= host_b <= 14 * N + 4 * 256 * len(sizes)
    dev_b2, _ = S.slide_state_bytes(sizes + [5_000_000] * 7, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    assert dev_b2 == dev_b
    free0, _ = torch.cuda.mem_get_info()
    st = S.slide_state_create(sizes, R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    try:
        free1, _ = torch.cuda.mem_get_info()
        assert dev_b <= free0 - free1 <= dev_b + (64 << 20)
    finally:
        S.slide_state_destroy(st)


def _mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def _host_view(ptr, n, ctype, dtype):
    """numpy view (no copy) of n values of pinned host memory owned by the state."""
    return np.ctypeslib.as_array((ctype * n).from_address(ptr)).view(dtype)


@pytest.mark.parametrize("name", ["h8192x8_streamed", "h5120x40_streamed"])
def test_streamed_full_size_sampled(S, name):
    """The full host-streamed workloads, sampled: every checked unit's sampled
    elements against the oracle after each step; the BF16 copy equals bf16 of
    the master; t advanced once per step.  Also every element of one whole
    unit (878M parameters of the h8192 model, 330M of the h5120 one).  The 40-layer h5120 model (14.8 B
    parameters) keeps its BF16 copy in HBM so that its 12 B/param of FP32
    state fits the host; the sampled elements are read through views of the
    pinned state, without copying it."""
    w = W.ALL[name]()
    sizes = [u.numel for u in w.units]
    flags = S.SLIDE_FLAG_BF16_COPY_IN_HBM if name == "h5120x40_streamed" else 0
    _, host_b = S.slide_state_bytes(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)
    # one whole unit is also checked on every element: its replicas and the
    # oracle's state of that unit live in ordinary host memory beside the pins
    whole = len(w.units) // 2
    extra = (2 * w.R + 14) * sizes[whole]
    if _mem_available() < host_b + extra + (16 << 30):
        pytest.skip(f"host memory: needs {(host_b + extra) / 2**30:.0f} GiB + 16 GiB headroom, "
                    f"{_mem_available() / 2**30:.0f} GiB available")
    st = S.slide_state_create(sizes, w.R, residency=S.SLIDE_RESIDENCY_HOST_STREAMED, flags=flags)
    try:
        for ui, u in enumerate(w.units):
            th_p = S.slide_layer_ptrs(st, ui)[0]
            synth.dev_master(th_p, u.numel, w.seed, unit=ui)
        torch.cuda.synchronize()
        check_units = sorted({0, len(w.units) // 2, len(w.units) - 1})
        samples = {}
        for ui in check_units:
            u = w.units[ui]
            idx = pu.sample_indices(u.numel, 50_000, seed=ui)
            samples[ui] = [idx, synth.gather_master(idx, w.seed, unit=ui), np.zeros(idx.size, np.float32),
                           np.zeros(idx.size, np.float32)]
        hp = S.hparams(*w.hparams_tuple())
        for t in range(1, w.steps + 1):
            holder = ModelGradsHolder(w, t)
            S.slide_model_step_streamed(st, synth.grad_fn_address(), holder.mg, hp)
        for ui in check_units:
            idx, th, m, v = samples[ui]
            wb = pu.oracle_sampled(w, ui, idx, 1, w.steps, th, m, v)
            n = w.units[ui].numel
            pt, pm, pv, pw = S.slide_layer_ptrs(st, ui)
            a = _host_view(pt, n, C.c_float, np.float32)[idx].copy()
            b = _host_view(pm, n, C.c_float, np.float32)[idx].copy()
            c = _host_view(pv, n, C.c_float, np.float32)[idx].copy()
            wg = np.empty(n, np.uint16)
            assert S.slide_layer_get(st, ui, bf16=wg) == w.steps
            wg = wg[idx]
            rep = [pu.compare_fp32("theta", a, th), pu.compare_fp32("m", b, m),
                   pu.compare_fp32("v", c, v), pu.compare_bf16("w", wg, wb)]
            pu.assert_parity(rep)
            assert all(r["not_bit_equal"] == 0 for r in rep)
            assert np.array_equal(wg, oracle.f32_to_bf16(a))
        assert all(S.slide_layer_get(st, ui) == w.steps for ui in range(len(w.units)))
        check_whole_unit(S, st, w, whole, bf16_in_hbm=bool(flags & S.SLIDE_FLAG_BF16_COPY_IN_HBM))
    finally:
        S.slide_state_destroy(st)


def check_whole_unit(S, st, w, ui, bf16_in_hbm=False):
    """Every element of unit ui of a host-streamed state after w.steps steps
    against the oracle over the whole unit (inputs from the seeded generator,
    the same values that the streamed step's gradient callback produced)."""
    n = w.units[ui].numel
    hp_or = pu.hp_oracle(w)
    th = pu.master_threaded(n, w.seed, unit=ui)
    m, v, wb = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    bufs = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(w.R)]
    for t in range(1, w.steps + 1):
        for r in range(w.R):
            pu.unit_grad_dev(w, ui, t, r, bufs[r].data_ptr())
        reps = pu.replicas_to_host(w, ui, t, bufs, n)
        pu.oracle_step_threaded(reps, th, m, v, wb, hp_or, t)
        del reps
    del bufs
    pt, pm, pv, pw = S.slide_layer_ptrs(st, ui)
    a = _host_view(pt, n, C.c_float, np.float32)
    b = _host_view(pm, n, C.c_float, np.float32)
    c = _host_view(pv, n, C.c_float, np.float32)
    if bf16_in_hbm:   # the BF16 copy is device memory: copy it out
        wg = np.empty(n, np.uint16)
        S.slide_layer_get(st, ui, bf16=wg)
    else:
        wg = _host_view(pw, n, C.c_uint16, np.uint16)
    rep = [pu.compare_fp32_all(f"theta unit {ui}", a, th), pu.compare_fp32_all(f"m unit {ui}", b, m),
           pu.compare_fp32_all(f"v unit {ui}", c, v), pu.compare_bf16_all(f"w unit {ui}", wg, wb)]
    print(rep)
    pu.assert_parity(rep)
    assert all(r["not_bit_equal"] == 0 for r in rep), rep
