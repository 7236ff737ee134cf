"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching the
device.  Valid calls on a machine without a GB300 fail with
LP_ERR_UNSUPPORTED_DEVICE: there is no fallback path.
"""

import ctypes

import pytest
import torch

from invariant_token_logprobs_gb300 import lp

OK, INVALID, MISALIGNED, UNSUPPORTED, WS_SMALL = 0, 1, 2, 3, 4
A = 1 << 20  # a fake, well-aligned device address; never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    return lp.load()


def test_exports_every_declared_symbol(lib):
    names = lp.declared_symbols()
    assert len(names) == 31
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lp._SIGNATURES)


def test_status_strings_and_backend(lib):
    for code, name in lp.STATUS.items():
        assert lp.lp_status_string(code) == name
    assert lp.lp_status_string(99) == "LP_ERR_UNKNOWN"
    assert lp.lp_backend_id() == "lp.sm103a.bitwise.v1"


def test_vocab_shard_range():
    V = 151936
    assert lp.vocab_shard_range(V, 0, 1) == (0, V)
    assert lp.vocab_shard_range(V, 1, 2) == (75968, V)
    assert [lp.vocab_shard_range(V, i, 4) for i in range(4)] == [
        (0, 37984), (37984, 75968), (75968, 113952), (113952, 151936)]
    # quarters of a vocabulary not divisible by 4: floor(q V / 4)
    assert [lp.vocab_shard_range(10, i, 4) for i in range(4)] == [(0, 2), (2, 5), (5, 7), (7, 10)]
    assert lp.vocab_shard_range(10, 1, 2) == (5, 10)
    for bad in [(V, 0, 3), (V, 2, 2), (V, -1, 4), (0, 0, 1)]:
        with pytest.raises(lp.LpError):
            lp.vocab_shard_range(*bad)


def test_workspace_sizes(lib):
    # header + one 16-byte state per row and 256-column tile of each quarter
    tiles = -(-(151936 // 4) // 256)
    assert tiles == 149
    assert lp.lp_linear_logprob_workspace_size(512, 4096, 151936) == 256 + 4 * tiles * 512 * 16
    assert lp.lp_linear_logprob_partials_workspace_size(512, 4096, 151936, 2) == 256 + 2 * tiles * 512 * 16
    assert lp.lp_linear_logprob_workspace_size(0, 8, 10) == 256
    # fewer than 16 rows: a 16-row bf16 copy of H follows, 256-byte aligned
    t1000 = -(-((1000 + 3) // 4) // 256)  # tiles per quarter of V = 1000
    assert lp.lp_linear_logprob_workspace_size(5, 64, 1000) == \
        -(-(256 + 4 * t1000 * 5 * 16) // 256) * 256 + 16 * 64 * 2
    assert lp.lp_linear_logprob_workspace_size(16, 64, 1000) == 256 + 4 * t1000 * 16 * 16
    # the copy's rows are d rounded up to 8 wide
    assert lp.lp_linear_logprob_workspace_size(5, 60, 1000) == \
        -(-(256 + 4 * t1000 * 5 * 16) // 256) * 256 + 16 * 64 * 2
    assert lp.lp_linear_logprob_workspace_size(-1, 8, 10) == 0
    assert lp.lp_linear_logprob_workspace_size(5, 0, 10) == 0  # no hidden size


def test_logits_argument_errors(lib):
    f = lib.lp_logprob_from_logits
    assert f(A, 100, A, 0, 100, A, A, None) == OK          # T == 0: nothing to do
    assert f(A, 100, A, -1, 100, A, A, None) == INVALID
    assert f(A, 100, A, 4, 0, A, A, None) == INVALID       # V == 0
    assert f(A, 99, A, 4, 100, A, A, None) == INVALID      # ld < V
    assert f(None, 100, A, 4, 100, A, A, None) == INVALID
    assert f(A, 100, None, 4, 100, A, A, None) == INVALID
    assert f(A, 100, A, 4, 100, None, A, None) == INVALID
    assert f(A + 2, 100, A, 4, 100, A, A, None) == MISALIGNED
    assert f(A, 100, A + 4, 4, 100, A, A, None) == MISALIGNED
    assert f(A, 100, A, 4, 100, A + 1, A, None) == MISALIGNED


def test_fused_argument_errors(lib):
    f = lib.lp_linear_logprob
    ws = lp.lp_linear_logprob_workspace_size(64, 256, 8192)
    args = [A, 256, A, 256, A, 64, 256, 8192, A, A, A, ws, None]

    def call(**kw):
        a = list(args)
        for k, v in kw.items():
            a[["H", "ld_h", "W", "ld_w", "y", "T", "d", "V", "logp", "ent", "ws", "wsb", "s"].index(k)] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(d=0) == INVALID
    assert call(V=0) == INVALID
    assert call(ld_h=255) == INVALID
    assert call(H=None) == INVALID
    assert call(logp=None) == INVALID
    assert call(ws=None) == INVALID
    assert call(H=A + 8) == MISALIGNED
    assert call(W=A + 2) == MISALIGNED
    assert call(ld_h=260) == MISALIGNED      # row pitch not a multiple of 16 bytes
    assert call(ws=A + 128) == MISALIGNED
    assert call(wsb=ws - 1) == WS_SMALL
    g = lib.lp_linear_logprob_partials
    wsp = lp.lp_linear_logprob_partials_workspace_size(64, 256, 8192, 4)
    assert g(A, 256, A, 256, A, 64, 256, 8192, 4, 4, A, A, wsp, None) == INVALID  # shard index
    assert g(A, 256, A, 256, A, 64, 256, 8192, 0, 3, A, A, wsp, None) == INVALID  # 3 shards
    assert g(A, 256, A, 256, A, 64, 256, 8192, 1, 4, A + 4, A, wsp, None) == MISALIGNED
    assert g(A, 256, A, 256, A, 64, 256, 8192, 1, 4, A, A, wsp - 16, None) == WS_SMALL


def test_temperature_argument_errors(lib):
    f = lib.lp_logprob_from_logits_temperature
    for bad in (0.0, -0.7, float("nan"), float("inf"), 1e-45):
        assert f(A, 100, A, 4, 100, bad, A, A, None) == INVALID, bad
    assert f(A, 100, A, 0, 100, 0.7, A, A, None) == OK
    g = lib.lp_linear_logprob_temperature
    ws = lp.lp_linear_logprob_workspace_size(64, 256, 8192)
    assert g(A, 256, A, 256, A, 64, 256, 8192, -1.0, A, A, A, ws, None) == INVALID
    assert g(A, 256, A, 256, A, 64, 256, 8192, 0.7, A, A, A, ws - 1, None) == WS_SMALL


def test_backward_argument_errors(lib):
    f = lib.lp_linear_logprob_backward
    ws = lp.lp_linear_logprob_backward_workspace_size(64, 256, 8192)
    assert ws > lp.lp_linear_logprob_workspace_size(64, 256, 8192)
    #       H  ldh  W  ldw y  T   d    V     tau  lse ent gl ge gH gW ws  wsb stream
    base = [A, 256, A, 256, A, 64, 256, 8192, 1.0, A, A, A, A, A, A, A, ws, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return f(*a)

    assert f(*base[:5], 0, *base[6:]) == OK          # T == 0
    assert call(8, 0.0) == INVALID                    # temperature
    assert call(13, None) == INVALID                  # grad_H
    assert call(9, None) == INVALID                   # lse without entropy
    a = list(base); a[11] = None; a[12] = None
    assert f(*a) == INVALID                           # no upstream gradient
    assert call(13, A + 4) == MISALIGNED              # grad_H 16-byte aligned
    assert call(16, ws - 1) == WS_SMALL
    assert lp.lp_linear_logprob_backward_workspace_size(-1, 8, 8) == 0
    # the _ex form: grad_W written as float32 (0) or bf16 (1), or added into (2)
    ex = lib.lp_linear_logprob_backward_ex
    assert ex(*base[:15], 3, *base[15:]) == INVALID
    assert ex(*base[:15], -1, *base[15:]) == INVALID
    assert ex(*base[:5], 0, *base[6:15], 2, *base[15:]) == OK  # T == 0


def _backward_ws(T, d, V, V_total):
    # header + quarter states, log Z / logp / entropy, bf16 G [T, round8(V)], and the
    # partial grad_H: 28 of them when V_total % 64 == 0 (7 per quarter), else 19
    a = lambda x: -(-x // 256) * 256
    tiles = -(-((V_total + 3) // 4) // 256)
    # a shard has its statistics given: no forward workspace, only the header
    o = a(256 + 4 * tiles * T * 16 if V == V_total else 256) + 3 * a(4 * T)
    o += a(2 * T * (-(-V // 8) * 8))
    return o + a(4 * (28 if V_total % 64 == 0 else 19) * T * d)


def test_backward_workspace_layout(lib):
    assert lp.lp_linear_logprob_backward_workspace_size(64, 256, 8192) == _backward_ws(64, 256, 8192, 8192)
    assert lp.lp_linear_logprob_backward_workspace_size(64, 256, 8200) == _backward_ws(64, 256, 8200, 8200)
    for n in (1, 2, 4):
        assert lp.lp_linear_logprob_partials_backward_workspace_size(512, 4096, 151936, n) == \
            _backward_ws(512, 4096, 151936 // n, 151936)
    # one shard: the whole vocabulary, any V
    assert lp.lp_linear_logprob_partials_backward_workspace_size(64, 256, 8200, 1) == \
        lp.lp_linear_logprob_backward_workspace_size(64, 256, 8200)
    assert lp.lp_linear_logprob_partials_backward_workspace_size(64, 256, 8192, 3) == 0
    assert lp.lp_linear_logprob_partials_backward_workspace_size(-1, 256, 8192, 2) == 0


def test_shard_backward_argument_errors(lib):
    f = lib.lp_linear_logprob_partials_backward
    ws = lp.lp_linear_logprob_partials_backward_workspace_size(64, 256, 8192, 2)
    #       H  ldh  W  ldw y  T   d    Vtot  i  n  tau  lse ent gl ge gH gW dt ws  wsb stream
    base = [A, 256, A, 256, A, 64, 256, 8192, 1, 2, 1.0, A, A, A, A, A, A, 0, A, ws, None]

    def call(**kw):
        idx = dict(H=0, T=5, V=7, i=8, n=9, tau=10, lse=11, ent=12, gl=13, ge=14, gH=15, gW=16,
                   dt=17, ws=18, wsb=19)
        a = list(base)
        for k, v in kw.items():
            a[idx[k]] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(i=2) == INVALID                     # shard index
    assert call(n=3) == INVALID                     # shard count
    assert call(V=8200) == INVALID                  # quarters not on 16-column boundaries
    assert call(lse=None) == INVALID                # a shard needs the merged statistics
    assert call(ent=None) == INVALID
    assert call(gl=None, ge=None) == INVALID        # no upstream gradient
    assert call(dt=3) == INVALID                    # grad_W dtype (0, 1, 2 are valid)
    assert call(tau=0.0) == INVALID
    assert call(gH=None) == INVALID
    assert call(gH=A + 8) == MISALIGNED
    assert call(wsb=ws - 1) == WS_SMALL
    g = lib.lp_merge_grad_h_partials
    arr = (ctypes.c_void_p * 4)(A, A, A, A)
    assert g(arr, 3, 8, 256, A, None) == INVALID
    assert g(arr, 4, 0, 256, A, None) == OK
    assert g(arr, 4, 8, 252, A, None) == MISALIGNED  # d % 8
    bad = (ctypes.c_void_p * 2)(A, A + 8)
    assert g(bad, 2, 8, 256, A, None) == MISALIGNED
    none = (ctypes.c_void_p * 2)(A, None)
    assert g(none, 2, 8, 256, A, None) == INVALID
    assert g(arr, 2, 8, 256, A + 4, None) == MISALIGNED


def test_merge_argument_errors(lib):
    f = lib.lp_merge_partials
    arr = (ctypes.c_void_p * 4)(A, A, A, A)
    assert f(arr, 3, 8, A, A, None) == INVALID
    assert f(arr, 4, 0, A, A, None) == OK
    bad = (ctypes.c_void_p * 2)(A, A + 8)
    assert f(bad, 2, 8, A, A, None) == MISALIGNED
    none = (ctypes.c_void_p * 2)(A, None)
    assert f(none, 2, 8, A, A, None) == INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gb300_fails_loudly(lib):
    assert lib.lp_logprob_from_logits(A, 100, A, 4, 100, A, A, None) == UNSUPPORTED
    assert lib.lp_logprob_from_logits_lse(A, 100, A, 4, 100, ctypes.c_float(1.0), A, A, A,
                                          None) == UNSUPPORTED
    G = A + (1 << 16)
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, ctypes.c_float(1.0), A, A, A,
                                               None, G, 100, None) == UNSUPPORTED
    ws = lp.lp_linear_logprob_workspace_size(64, 256, 8192)
    assert lib.lp_linear_logprob(A, 256, A, 256, A, 64, 256, 8192, A, A, A, ws, None) == UNSUPPORTED
    arr = (ctypes.c_void_p * 1)(A)
    assert lib.lp_merge_partials(arr, 1, 8, A, A, None) == UNSUPPORTED
    assert lib.lp_merge_partials_lse(arr, 1, 8, A, A, A, None) == UNSUPPORTED
    assert lib.lp_logprob_partials_from_logits_backward(A, 100, A, 4, 200, 1, 2, ctypes.c_float(1.0),
                                                        A, A, A, None, A + (1 << 16), 100,
                                                        None) == UNSUPPORTED
    # a shard index outside [0, n_shards) is an argument error before any device check
    assert lib.lp_logprob_partials_from_logits_backward(A, 100, A, 4, 200, 2, 2, ctypes.c_float(1.0),
                                                        A, A, A, None, A + (1 << 16), 100,
                                                        None) == INVALID
    wsb = lp.lp_linear_logprob_partials_backward_workspace_size(64, 256, 8200, 1)
    assert lib.lp_linear_logprob_partials_backward(A, 256, A, 256, A, 64, 256, 8200, 0, 1,
                                                   ctypes.c_float(1.0), A, A, A, None, A, A, 0,
                                                   A, wsb, None) == UNSUPPORTED
    assert lib.lp_merge_grad_h_partials(arr, 1, 8, 256, A, None) == UNSUPPORTED
    assert lib.lp_set_persistent_grid_limit(-1) == INVALID
    assert lib.lp_set_persistent_grid_limit(0) == OK
    assert lib.lp_set_fault_injection(3) == INVALID
    assert lib.lp_set_fault_injection(-1) == INVALID
    assert lib.lp_set_fault_injection(2) == OK
    assert lib.lp_set_fault_injection(0) == OK


def test_logits_backward_argument_checks(lib):
    f = ctypes.c_float(1.0)
    G = A + (1 << 16)
    # no upstream gradient, no saved statistics, a short row stride, overlap
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, f, A, A, None, None, G, 100,
                                               None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, f, None, A, A, None, G, 100,
                                               None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, f, A, A, A, None, G, 99,
                                               None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, f, A, A, A, None, A + 396, 100,
                                               None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, ctypes.c_float(0.0), A, A, A,
                                               None, G, 100, None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 4, 100, f, A, A, A + 2, None, G, 100,
                                               None) == MISALIGNED
    assert lib.lp_logprob_from_logits_lse(A, 100, A, 4, 100, f, A, A, None, None) == INVALID
    assert lib.lp_logprob_from_logits_backward(A, 100, A, 0, 100, f, None, None, None, None, None,
                                               100, None) == OK
