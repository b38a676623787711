"""Host-side tests of the C-ABI library (no GPU needed): it loads, exports every
entry point include/slide.h declares, validates configurations before
touching a device, and its byte accounting follows the 16N-byte state of
mixed-precision Adam ("SlideDP: Scaling Host-Resident LLM Fine-Tuning Across
Multiple GPUs", Prerequisites: BF16 weights 2N + BF16 gradients 2N + FP32
master 4N + FP32 Adam moments 8N) and the 12 = 4 + 4 + 4 bytes of FP32 state
per parameter ("Accelerating the Training of Large Language Models using
Efficient Activation Rematerialization and Optimal Hybrid Parallelism",
section 3, memory footprint item 2).
"""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def S():
    import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
    from mixed_precision_adam_grad_gb300 import build
    build.build()
    import mixed_precision_adam_grad_gb300 as S
    return S


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"SLIDE_API[^;(]*?\b(slide_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol(S):
    names = declared_symbols()
    assert {"slide_state_create", "slide_layer_step", "slide_model_step_streamed",
            "slide_state_destroy"} <= set(names), names
    lib = C.CDLL(S.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert S.slide_abi_version() == 2


def test_every_entry_point_cites_its_passage():
    """Each exported call's comment in include/*.h names the passage that
    defines it (page title and section), or says that the pages have none."""
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        for m in re.finditer(r"SLIDE_API[^;(]*?\b(slide_\w+)\s*\(", text):
            # the comment block directly above the declaration
            before = text[:m.start()].rstrip()
            assert before.endswith("*/"), f"{m.group(1)} has no comment block"
            block = re.sub(r"\s*\n\s*\*\s?", " ", before[before.rfind("/*"):])
            cites = re.search(r"Defined by:|has\s+no counterpart|no\s+passage", block)
            assert cites, f"{m.group(1)}: its comment cites no passage"
            if "Defined by:" in block and "no passage" not in block:
                names = ("SlideDP", "Heterogeneous Co-Design", "Accelerating the", "passage cited above",
                         "same passages as")
                assert any(n in block for n in names), f"{m.group(1)}: no page title in its citation"


def test_binding_fails_loudly_without_library(S, monkeypatch):
    from mixed_precision_adam_grad_gb300 import _binding
    monkeypatch.setattr(_binding, "LIB_PATH", os.path.join(ROOT, "no_such_libslide.so"))
    with pytest.raises(ImportError):
        _binding._load()


A = 256


def al(x):
    return (x + A - 1) // A * A


def test_accounting_16N(S):
    """Per parameter the library holds 4 (master) + 4 + 4 (m, v) + 2 (BF16
    copy) bytes; with the 2 bytes of one BF16 gradient that the caller holds
    this is the pages' 16 bytes per parameter."""
    sizes = [100_930_560, 1, 17, 0]
    dev, host = S.slide_state_bytes(sizes, 4)
    scratch = al(8 * 4096) + A
    assert host == 0
    assert dev == sum(3 * al(4 * n) + al(2 * n) for n in sizes) + len(sizes) * scratch
    N = sum(sizes)
    state_per_param = 4 + 4 + 4 + 2
    assert state_per_param + 2 == 16              # + one BF16 gradient replica
    assert 4 + 4 + 4 == 12                        # FP32 master + two Adam moments
    assert state_per_param * N <= dev - len(sizes) * scratch <= state_per_param * N + 4 * A * len(sizes)


def test_accounting_host_inputs_staging(S):
    """SLIDE_FLAG_HOST_INPUTS adds two staging sets of R replicas of the
    largest layer (BF16, or FP32 with SLIDE_FLAG_FP32_GRADS)."""
    sizes = [1000, 70001, 17]
    for R, fp32, g in ((3, False, 2), (4, True, 4)):
        f = S.SLIDE_FLAG_FP32_GRADS if fp32 else 0
        base, _ = S.slide_state_bytes(sizes, R, flags=f)
        with_in, host = S.slide_state_bytes(sizes, R, flags=f | S.SLIDE_FLAG_HOST_INPUTS)
        assert host == 0
        assert with_in - base == 2 * R * al(g * max(sizes))


def test_accounting_streamed_window_independent_of_N(S):
    one = [330_311_680]
    many = [778_567_680] + [330_311_680] * 40 + [778_567_680]
    d1, h1 = S.slide_state_bytes([778_567_680] + one, 4, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    d2, h2 = S.slide_state_bytes(many, 4, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    assert d1 == d2                                    # window: two slots of the largest unit
    N = sum(many)
    assert N == 14_769_602_560
    assert 14 * N <= h2 <= 14 * N + 4 * A * len(many)  # master, m, v, BF16 mirror
    R, maxn = 4, 778_567_680
    slot = 3 * al(4 * maxn) + al(2 * maxn) * (1 + R) + al(8 * 4096) + A
    assert d2 == 2 * slot


def test_accounting_streamed_bf16_copy_in_hbm(S):
    """With the BF16 copy in HBM the host holds 12 B/param (FP32 master and
    two moments); the device holds 2 B/param of BF16 copy and the window
    drops its two BF16 slots (the update writes the resident copy in place)."""
    many = [778_567_680] + [330_311_680] * 40 + [778_567_680]
    N = sum(many)
    d0, h0 = S.slide_state_bytes(many, 4, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    d1, h1 = S.slide_state_bytes(many, 4, residency=S.SLIDE_RESIDENCY_HOST_STREAMED,
                                 flags=S.SLIDE_FLAG_BF16_COPY_IN_HBM)
    assert 12 * N <= h1 <= 12 * N + 3 * A * len(many)
    assert d1 == d0 + sum(al(2 * n) for n in many) - 2 * al(2 * max(many))
    assert h0 - h1 == sum(al(2 * n) for n in many)


@pytest.mark.parametrize("kw,msg", [
    (dict(layer_numel=[10], n_replicas=0), "n_replicas"),
    (dict(layer_numel=[10], n_replicas=9), "n_replicas"),
    (dict(layer_numel=[-1], n_replicas=1), "layer_numel"),
    (dict(layer_numel=[10], n_replicas=1, residency=7), "residency"),
    (dict(layer_numel=[10], n_replicas=1, chunk_bytes=100), "chunk_bytes"),
    (dict(layer_numel=[10], n_replicas=1, window_layers=3), "window_layers"),
    (dict(layer_numel=[10], n_replicas=1, flags=64), "flag"),
    (dict(layer_numel=[10], n_replicas=1, residency=1, flags=32), "HBM residency"),
    (dict(layer_numel=[], n_replicas=1), "n_layers"),
    (dict(layer_numel=[10], n_replicas=1, chunk_bytes_d2h=100), "chunk_bytes_d2h"),
    (dict(layer_numel=[1 << 26], n_replicas=1, residency=1, chunk_bytes=1024), "65536 chunks"),
    (dict(layer_numel=[1 << 26], n_replicas=1, residency=1, chunk_bytes_d2h=2048), "65536 chunks"),
    (dict(layer_numel=[10], n_replicas=1, host_arena=1 << 20, host_arena_bytes=1 << 20), "streamed residency"),
    (dict(layer_numel=[10], n_replicas=1, residency=1, host_arena=(1 << 20) + 16, host_arena_bytes=1 << 20),
     "256-byte"),
    (dict(layer_numel=[10], n_replicas=1, residency=1, host_arena_bytes=1 << 20), "without a host_arena"),
    (dict(layer_numel=[10], n_replicas=1, residency=1, flags=16, host_arena=1 << 20, host_arena_bytes=1 << 20),
     "exclude"),
])
def test_config_validation_without_gpu(S, kw, msg):
    numel = kw.pop("layer_numel")
    R = kw.pop("n_replicas")
    for fn in (S.slide_state_bytes, S.slide_state_create):
        with pytest.raises(S.SlideError) as e:
            fn(numel, R, **kw)
        assert e.value.status == S.SLIDE_ERR_INVALID_ARG
        assert msg in str(e.value)


def test_null_state_is_rejected(S):
    lib = S.lib
    assert lib.slide_layer_status(None, 0) == S.SLIDE_ERR_INVALID_ARG
    assert "NULL" in S.slide_last_error()
    lib.slide_state_destroy(None)  # NULL-safe
