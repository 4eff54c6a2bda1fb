"""Host-side checks of the C ABI: the library builds for sm_103a, loads, and
exports every entry point that include/sanatan.h declares; argument checks that
fail before any device work return their status codes.  No kernel runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sanatan.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SANATAN_API\s+[\w\s\*]*?\b(sanatan_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from constant_state_recurrence_gb300 import build, sanatan
    build.build(quiet=True)
    return sanatan.lib()


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for name in ("sanatan_featurize", "sanatan_chunk_fwd", "sanatan_chunk_bwd",
                 "sanatan_decode_step"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    handle = ctypes.CDLL(lib._name)
    for name in declared_symbols():
        assert hasattr(handle, name), name


def test_binding_covers_every_declared_symbol():
    from constant_state_recurrence_gb300 import sanatan
    assert set(declared_symbols()) <= set(sanatan.exported_symbols())


def test_state_bytes_matches_the_pages(lib):
    import oracle_pins as P
    g = P.read_golden("memory_accounting.txt")
    assert lib.sanatan_state_bytes(12, 12, 64, 64) == int(g["state_bytes_total"][0][0])
    assert lib.sanatan_state_bytes(1, 1, 64, 64) == int(g["state_bytes_per_head"][0][0])


def test_status_strings(lib):
    for s in range(6):
        assert lib.sanatan_status_string(s)
    assert lib.sanatan_abi_version() >= 1


def test_argument_errors_before_any_launch(lib):
    P = ctypes.c_void_p
    # bad dtype enum
    assert lib.sanatan_featurize(None, 7, None, None, None, 1, 1, 1, 64, 0, None, 0, None) == 1
    # unsupported head size
    assert lib.sanatan_featurize(None, 0, None, None, None, 1, 1, 1, 32, 0, None, 0, None) == 2
    # empty problem is a no-op
    assert lib.sanatan_featurize(None, 0, None, None, None, 0, 1, 1, 64, 0, None, 0, None) == 0
    # misaligned pointer
    assert lib.sanatan_featurize(P(8), 0, P(16), P(16), P(16), 1, 1, 1, 64, 0, P(32), 0, None) == 1
    # S0 without z0
    assert lib.sanatan_chunk_fwd(P(16), P(16), P(16), 1, P(16), P(16), P(16), 1, 1, 4, 64, 64, 0,
                                 0.0, P(16), None, P(16), None, None, None, None, 0, None) == 1
    # negative sizes, unsupported dv
    assert lib.sanatan_chunk_fwd(None, None, None, 1, None, None, None, -1, 1, 4, 64, 64, 0, 0.0,
                                 None, None, None, None, None, None, None, 0, None) == 1
    assert lib.sanatan_chunk_fwd(None, None, None, 1, None, None, None, 1, 1, 4, 64, 32, 0, 0.0,
                                 None, None, None, None, None, None, None, 0, None) == 2
    # decode: G must be positive; null state
    assert lib.sanatan_decode_step(None, None, None, None, None, None, None, None, None, 4, 0, 64,
                                   64, 0.0, None, None) == 1
    assert lib.sanatan_decode_step(None, P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                                   4, 4, 64, 64, 0.0, P(16), None) == 1
    # power attention: p below 1, p above the largest supported, misaligned D
    assert lib.sanatan_power_fwd(None, None, None, None, None, None, 1, 1, 4, 64, 64, 0, 0, 0.0,
                                 None, None, None, 0, None) == 1
    assert lib.sanatan_power_fwd(None, None, None, None, None, None, 1, 1, 4, 64, 64, 0, 9, 0.0,
                                 None, None, None, 0, None) == 2
    assert lib.sanatan_power_fwd(P(16), P(16), P(16), P(16), P(16), P(16), 1, 1, 4, 64, 64, 0, 2,
                                 0.0, P(16), P(8), P(16), 1 << 20, None) == 1
    # empty problems are no-ops; a short workspace is rejected
    assert lib.sanatan_power_fwd(None, None, None, None, None, None, 1, 1, 0, 64, 64, 0, 2, 0.0,
                                 None, None, None, 0, None) == 0
    need = lib.sanatan_power_fwd_workspace_size(1, 1, 4, 64, 64)
    assert lib.sanatan_power_fwd(P(16), P(16), P(16), P(16), P(16), P(16), 1, 1, 4, 64, 64, 0, 2,
                                 0.0, P(16), None, P(16), need - 16, None) == 1


def test_power_workspace_size(lib):
    # bf16 Phi(q), Phi(k) (320 non-constant features each) and [v | 1 | 0] per token,
    # whole 128-token chunks
    per_chunk = 128 * (2 * 320 + 80) * 2
    assert lib.sanatan_power_fwd_workspace_size(1, 1, 1, 64, 64) == per_chunk
    assert lib.sanatan_power_fwd_workspace_size(4, 12, 2048, 64, 64) == 48 * 16 * per_chunk
    assert lib.sanatan_power_fwd_workspace_size(2, 3, 129, 64, 64) == 6 * 2 * per_chunk
    assert lib.sanatan_power_fwd_workspace_size(1, 1, 0, 64, 64) == 0
    assert lib.sanatan_power_fwd_workspace_size(1, 1, 4, 32, 64) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from constant_state_recurrence_gb300 import sanatan
    monkeypatch.setattr(sanatan, "_lib", None)
    monkeypatch.setattr(sanatan, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        sanatan.lib()


def test_selftest_probe_rejects_bad_limits_before_any_launch(lib):
    assert lib.sanatan_selftest_wait_timeout(10, 0, None) == 1             # below 1 us
    assert lib.sanatan_selftest_wait_timeout(2 * 10**9, 0, None) == 1      # above 1 s
    assert lib.sanatan_selftest_wait_timeout(10**6, 2, None) == 1          # bad flag


def test_ablation_argument_errors_before_any_launch(lib):
    P = ctypes.c_void_p
    args = lambda p, ch, sh: (None, None, None, None, None, None, 1, 1, 8, 64, 64, 0, p, ch,  # noqa
                              sh, 0.0, None, None, None, 0, None)
    assert lib.sanatan_ablation_fwd(*args(2, 5, 0.0)) == 1      # channels
    assert lib.sanatan_ablation_fwd(*args(2, 4, 1.0)) == 1      # shift with four channels
    assert lib.sanatan_ablation_fwd(*args(2, 3, -1.0)) == 1     # negative shift
    assert lib.sanatan_ablation_fwd(*args(3, 3, 0.0)) == 2      # unsupported power
    del P


def test_eps_raw_conventions(lib):
    assert abs(lib.sanatan_eps_raw(1.0, 64, 0) - 256.000001) < 1e-4
    assert abs(lib.sanatan_eps_raw(2.0, 64, 1) - 5.12e-4) < 1e-9
    assert lib.sanatan_eps_raw(1.0, 0, 0) == -1.0 and lib.sanatan_eps_raw(1.0, 64, 2) == -1.0
    assert lib.sanatan_rate_from_raw(None, -1, 0.01, None, None) == 1
    assert lib.sanatan_rate_from_raw_bwd(None, None, -1, 0.01, None, None) == 1


def test_harmonic_state_bytes_and_argument_errors(lib):
    assert lib.sanatan_state_bytes_harmonic(12, 12, 64, 64, 1) == 14376960
    assert lib.sanatan_state_bytes_harmonic(12, 12, 64, 64, 2) == 12 * 12 * (640 * 64 + 640) * 4
    assert lib.sanatan_state_bytes_harmonic(1, 1, 64, 64, 0) == 0
    assert lib.sanatan_featurize_harmonic(None, 0, None, None, None, 1, 1, 1, 64, 0, 0, None, 0,
                                          None) == 1
    assert lib.sanatan_featurize_harmonic(None, 0, None, None, None, 1, 1, 1, 64, 0, 4, None, 0,
                                          None) == 2
