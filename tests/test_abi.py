"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, exports
every entry point declared in include/kda.h, and rejects bad arguments on the
host (before any launch) with the documented status codes."""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_18_gb300 as kda
from kimi_delta_attention_18_gb300._native import PrefillDesc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, TIMEOUT = range(6)


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    L = kda.lib()
    names = _declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(L, name), name


def test_status_strings_and_build_info():
    L = kda.lib()
    for s in range(6):
        assert L.kda_status_string(s)
    assert L.kda_status_string(99) == b"unknown status"
    assert b"sm_103a" in L.kda_build_info()


def _desc(**kw):
    base = dict(num_seqs=1, total_tokens=64, num_heads=2, dk=16, dv=16, act_dtype=0, chunk=16,
                num_segments=1)
    base.update(kw)
    return PrefillDesc(*[base[f] for f, _ in PrefillDesc._fields_])


def _prefill(desc, ptr=0x10000, ws=None, ws_len=0, cu=0x20000):
    L = kda.lib()
    p = ctypes.c_void_p(ptr) if ptr else None
    return L.kda_prefill_chunked(ctypes.byref(desc) if desc is not None else None, p, p, p, p, p,
                                 None, ctypes.c_void_p(cu) if cu else None, p, None,
                                 ctypes.c_void_p(ws) if ws else None, ws_len, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=8), UNSUPPORTED),
    (dict(dk=129), UNSUPPORTED),
    (dict(dv=0), INVALID),
    (dict(act_dtype=5), UNSUPPORTED),
    (dict(num_seqs=-1), INVALID),
    (dict(num_heads=0), INVALID),
    (dict(num_segments=-2), INVALID),
    (dict(num_segments=5000), UNSUPPORTED),
    # (sequence, head, segment) units must fit a grid dimension (below 2^31)
    (dict(num_seqs=1 << 20, num_heads=64, num_segments=64), UNSUPPORTED),
])
def test_prefill_rejects_bad_descriptor(kw, code):
    assert _prefill(_desc(**kw)) == code


def test_prefill_rejects_null_and_misaligned_pointers():
    L = kda.lib()
    assert L.kda_prefill_chunked(None, *([None] * 9), None, 0, None, None) == INVALID
    assert _prefill(_desc(), ptr=0) == INVALID          # q, k, ... missing
    assert _prefill(_desc(), ptr=0x10004) == INVALID    # not 16-byte aligned
    assert _prefill(_desc(), cu=0) == INVALID           # cu_seqlens missing
    assert _prefill(_desc(num_seqs=0)) == OK            # nothing to do, nothing launched


def test_timed_prefill_needs_its_four_events():
    L = kda.lib()
    p = ctypes.c_void_p(0x10000)
    args = [ctypes.byref(_desc()), p, p, p, p, p, None, ctypes.c_void_p(0x20000), p, None, None, 0,
            None]
    assert L.kda_prefill_chunked_timed(*args, None, None) == INVALID
    evs = (ctypes.c_void_p * 4)(0x1, 0x2, None, 0x4)
    assert L.kda_prefill_chunked_timed(*args, ctypes.cast(evs, ctypes.c_void_p), None) == INVALID


def test_prefill_split_requires_workspace():
    d = _desc(num_segments=4)
    need = kda.prefill_workspace_size(d)
    r256 = lambda b: (b + 255) // 256 * 256
    # (A, B, start) per (seq, head, segment) in fp32 + one dk-vector per token and head
    assert need == r256(1 * 2 * 4 * (16 * 16 + 2 * 16 * 16) * 4) + r256(64 * 2 * 16 * 4)
    # BF16 at dk = dv = 128 adds each start state's BF16 operand image (128 x 128)
    d2 = _desc(num_seqs=1, num_heads=8, total_tokens=4096, dk=128, dv=128, act_dtype=1,
               num_segments=9)
    need2 = kda.prefill_workspace_size(d2)
    assert need2 == (r256(1 * 8 * 9 * (128 * 128 + 2 * 128 * 128) * 4) +
                     r256(1 * 8 * 9 * 128 * 128 * 2) + r256(4096 * 8 * 128 * 2))
    assert _prefill(d) == WORKSPACE
    assert _prefill(d, ws=0x40000, ws_len=need - 1) == WORKSPACE
    assert _prefill(d, ws=0x40008, ws_len=need) == WORKSPACE  # misaligned workspace


def test_segment_choice():
    assert kda.prefill_num_segments(_desc(num_segments=7)) == 7
    # many chains: one pass each
    assert kda.prefill_num_segments(_desc(num_seqs=4, num_heads=128, total_tokens=4096,
                                          num_segments=0)) == 1
    # few long chains: split, at least 8 blocks per segment, at most 64 segments
    s = kda.prefill_num_segments(_desc(num_seqs=1, num_heads=8, total_tokens=4096, dk=128,
                                       dv=128, num_segments=0))
    assert 2 <= s <= 32
    s = kda.prefill_num_segments(_desc(num_seqs=1, num_heads=1, total_tokens=1 << 20,
                                       num_segments=0))
    assert s == 64
    assert kda.prefill_num_segments(_desc(chunk=4)) == 0
    assert kda.prefill_workspace_size(_desc(num_segments=1)) == 0


def test_decode_and_compose_host_checks():
    L = kda.lib()
    p = ctypes.c_void_p(0x10000)
    assert L.kda_decode_step(4, 2, 16, 18, 1, p, p, p, p, p, p, p, None, None) == UNSUPPORTED  # dv % 4
    assert L.kda_decode_step(4, 2, 256, 16, 1, p, p, p, p, p, p, p, None, None) == UNSUPPORTED
    assert L.kda_decode_step(4, 2, 16, 16, 3, p, p, p, p, p, p, p, None, None) == UNSUPPORTED
    assert L.kda_decode_step(4, 0, 16, 16, 1, p, p, p, p, p, p, p, None, None) == INVALID
    assert L.kda_decode_step(4, 2, 16, 16, 1, p, p, p, p, None, p, p, None, None) == INVALID
    assert L.kda_decode_step(4, 2, 16, 16, 1, p, p, p, p, ctypes.c_void_p(0x10002), p, p,
                             None, None) == INVALID
    # a misaligned status word is refused before anything is launched
    assert L.kda_decode_step(4, 2, 16, 16, 1, p, p, p, p, p, p, p, ctypes.c_void_p(0x10002),
                             None) == INVALID
    assert L.kda_decode_step(0, 2, 16, 16, 1, p, p, p, p, p, p, p, None, None) == OK
    assert L.kda_state_compose(2, 0, 16, 16, p, p, None, None, None, None, None, None) == INVALID
    assert L.kda_state_compose(2, 3, 16, 200, p, p, None, None, None, None, None, None) == UNSUPPORTED
    assert L.kda_state_compose(2, 3, 16, 16, None, p, None, None, None, None, None, None) == INVALID
    assert L.kda_state_compose(0, 3, 16, 16, None, None, None, None, None, None, None, None) == OK
    # start images exist only for dk = dv = 128 and must be 16-byte aligned
    assert L.kda_state_compose(2, 3, 16, 16, p, p, None, None, None, p, None, None) == INVALID
    assert L.kda_state_compose(2, 3, 128, 128, p, p, None, None, None,
                               ctypes.c_void_p(0x10008), None, None) == INVALID
    assert L.kda_state_compose(2, 3, 16, 16, p, p, None, None, None, None,
                               ctypes.c_void_p(0x10002), None) == INVALID
    d = _desc(num_segments=0)
    assert L.kda_state_transfer(ctypes.byref(d), 0, 1, None, p, p, p, p, p, p, p, None, None, None,
                                None) == INVALID
    assert L.kda_prefill_segments(ctypes.byref(d), 0, 1, p, p, p, p, p, None, p, p, None, None,
                                  None) == INVALID
    d = _desc(num_segments=4)
    for a, b in ((-1, 2), (3, 2), (0, 5)):
        assert L.kda_state_transfer(ctypes.byref(d), a, b, None, p, p, p, p, p, p, p, None, None,
                                    None, None) == INVALID
        assert L.kda_prefill_segments(ctypes.byref(d), a, b, p, p, p, p, p, None, p, p, None,
                                      None, None) == INVALID
    assert L.kda_state_transfer(ctypes.byref(d), 2, 2, None, p, p, p, p, p, p, p, None, None, None,
                                None) == OK
    # outputs need q, out_zero and out_transfer together
    assert L.kda_state_transfer(ctypes.byref(d), 0, 4, p, p, p, p, p, p, p, p, p, None, None,
                                None) == INVALID
    assert L.kda_prefill_combine(ctypes.byref(d), -1, p, None, p, p, p, None, None) == INVALID
    assert L.kda_prefill_combine(ctypes.byref(d), 0, None, None, p, p, p, None, None) == INVALID
    assert L.kda_prefill_combine(ctypes.byref(d), 4, None, None, None, None, None, None,
                                 None) == OK
    # start images only for BF16 at dk = dv = 128
    assert L.kda_prefill_combine(ctypes.byref(d), 0, p, p, p, p, p, None, None) == INVALID


def _prefill_ckpt(desc, interval, ckpt=0x50000, ws=None, ws_len=0):
    L = kda.lib()
    p = ctypes.c_void_p(0x10000)
    return L.kda_prefill_chunked_ckpt(ctypes.byref(desc), p, p, p, p, p, None,
                                      ctypes.c_void_p(0x20000), p, None, interval,
                                      ctypes.c_void_p(ckpt) if ckpt else None,
                                      ctypes.c_void_p(ws) if ws else None, ws_len, None, None)


def test_checkpoint_arguments_and_workspace():
    assert _prefill_ckpt(_desc(), 0) == INVALID         # interval required
    assert _prefill_ckpt(_desc(), 24) == INVALID        # not a multiple of 16
    assert _prefill_ckpt(_desc(), -16) == INVALID
    assert _prefill_ckpt(_desc(), 32, ckpt=0) == INVALID       # buffer missing
    assert _prefill_ckpt(_desc(), 32, ckpt=0x50002) == INVALID  # misaligned buffer
    L = kda.lib()
    d1 = _desc()  # one pass: no extra workspace
    assert L.kda_prefill_ckpt_workspace_size(ctypes.byref(d1), 32) == 0
    assert L.kda_prefill_ckpt_workspace_size(ctypes.byref(d1), 24) == 0   # invalid interval
    d = _desc(num_segments=4)  # split: + floor(T / interval) transfer matrices per head
    need = L.kda_prefill_ckpt_workspace_size(ctypes.byref(d), 32)
    r256 = lambda b: (b + 255) // 256 * 256
    assert need == kda.prefill_workspace_size(d) + r256((64 // 32) * 2 * 16 * 16 * 4)
    assert _prefill_ckpt(d, 32, ws=0x40000, ws_len=kda.prefill_workspace_size(d)) == WORKSPACE


def test_gated_prefill_host_checks():
    L = kda.lib()
    p = ctypes.c_void_p(0x10000)
    call = lambda d: L.kda_prefill_chunked_gated(ctypes.byref(d), p, p, p, p, p, None,
                                                 ctypes.c_void_p(0x20000), p, None, None, 0,
                                                 None, None)
    # the fused prologue runs in the BF16 d = 128 kernels only
    assert call(_desc()) == UNSUPPORTED
    assert call(_desc(act_dtype=1, dk=64, dv=64)) == UNSUPPORTED
    assert call(_desc(act_dtype=1, dk=128, dv=128, num_seqs=0)) == OK  # nothing to do
    d = _desc(act_dtype=1, dk=128, dv=128, num_segments=4)
    assert call(d) == WORKSPACE  # split needs the workspace of kda_prefill_workspace_size


def test_selftest_host_checks():
    L = kda.lib()
    assert L.kda_selftest_wait_timeout(0, ctypes.c_void_p(0x10000), None) == INVALID
    assert L.kda_selftest_wait_timeout(1000, None, None) == INVALID


def test_backward_host_checks():
    L = kda.lib()
    p = ctypes.c_void_p(0x10000)

    def call(d, ws=None, ws_len=0, g=p, cu=ctypes.c_void_p(0x20000), dq=p):
        return L.kda_prefill_backward(ctypes.byref(d), p, p, p, g, p, None, cu, p, None, dq, p,
                                      p, p, p, None, ctypes.c_void_p(ws) if ws else None,
                                      ws_len, None, None)

    d = _desc()
    need = L.kda_prefill_backward_workspace_size(ctypes.byref(d))
    # the state at every 4-token block start: [T/4 + N blocks][H][ceil(dv/8)][dk][8] fp32
    blocks = d.total_tokens // 4 + d.num_seqs
    assert need == blocks * d.num_heads * ((d.dv + 7) // 8) * d.dk * 8 * 4
    # segments: + A_s [dk][dk] and B_s, B^_s, X_s, Y_s [dk][dv] per (sequence, head, segment)
    d4 = _desc(num_segments=4)
    r256 = lambda b: (b + 255) // 256 * 256
    assert L.kda_prefill_backward_workspace_size(ctypes.byref(d4)) == r256(need) + \
        d4.num_seqs * d4.num_heads * 4 * (d4.dk * d4.dk + 4 * d4.dk * d4.dv) * 4
    assert L.kda_prefill_backward_workspace_size(ctypes.byref(_desc(chunk=32))) == 0
    assert L.kda_prefill_backward_num_segments(ctypes.byref(d4)) == 4
    assert L.kda_prefill_backward_num_segments(ctypes.byref(_desc(num_segments=500))) == 64
    assert L.kda_prefill_backward_num_segments(ctypes.byref(_desc(chunk=32))) == 0
    # BF16 at dk = dv = 128 takes the chunked backward, which splits sequences until
    # every SM has a one-chain CTA (at least 4 blocks per segment, at most 64) and keeps
    # BF16 states: [T/32][H] forward states (every 32 tokens) and [ceil(T/16) + N][H]
    # adjoints (every 16-token block) of 128 x 128 BF16, plus with S > 1 four 128 x 128
    # fp32 buffers per (sequence, head, segment), reused between the launches: the
    # forward states share their bytes with two of them
    for T, H, N in ((4096, 8, 1), (512, 8, 1), (64 * 512, 8, 64)):
        c = _desc(num_seqs=N, total_tokens=T, num_heads=H, dk=128, dv=128, act_dtype=1,
                  num_segments=0)
        S = L.kda_prefill_backward_num_segments(ctypes.byref(c))
        import torch  # the library counts the device's SMs, or assumes 148 without one
        sms = (torch.cuda.get_device_properties(0).multi_processor_count
               if torch.cuda.is_available() else 148)
        chains = N * H
        want_s = 1 if chains >= sms else max(1, min(-(-sms // chains), T // N // 16 // 4, 64))
        assert S == want_s, (T, H, N, S)
        img = 128 * 128 * 2
        fwd, seg = r256(T // 32 * H * img), r256(N * H * S * 128 * 128 * 4)
        want = r256(((T + 15) // 16 + N) * H * img)
        want += max(fwd, 2 * seg) + 2 * seg if S > 1 else fwd
        assert L.kda_prefill_backward_workspace_size(ctypes.byref(c)) == want
    # the chunked path moves rows as 16-byte pieces: unaligned rows are refused
    c = _desc(num_seqs=1, total_tokens=64, num_heads=2, dk=128, dv=128, act_dtype=1,
              num_segments=1)
    cneed = L.kda_prefill_backward_workspace_size(ctypes.byref(c))
    assert call(c, ws=0x40000, ws_len=cneed, g=ctypes.c_void_p(0x10004)) == INVALID
    assert call(d) == WORKSPACE
    assert call(d, ws=0x40000, ws_len=need - 1) == WORKSPACE
    assert call(d, ws=0x40008, ws_len=need) == WORKSPACE       # not 16-byte aligned
    assert call(d, ws=0x40000, ws_len=need, g=None) == INVALID  # input missing
    assert call(d, ws=0x40000, ws_len=need, dq=None) == INVALID  # output missing
    assert call(d, ws=0x40000, ws_len=need, dq=ctypes.c_void_p(0x10002)) == INVALID
    assert call(d, ws=0x40000, ws_len=need, cu=None) == INVALID
    assert call(_desc(num_seqs=0)) == OK  # nothing to do
    assert call(_desc(dk=256)) == UNSUPPORTED


def test_autograd_function_has_no_cpu_fallback():
    import torch
    from kimi_delta_attention_18_gb300.autograd import kda_prefill
    q = torch.zeros(16, 1, 16)
    with pytest.raises((ValueError, RuntimeError)):
        kda_prefill(q, q, q, q, torch.zeros(16, 1))
