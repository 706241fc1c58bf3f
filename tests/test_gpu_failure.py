"""The failure path of the fused decode stack, exercised without a fault.

The pages' TP serving hang modes are a collective that never completes
because one rank never arrives.  Here the stand-in for a rank is a CTA, and
the collective is a tile's split-K reduction: with the library's test hook a
CTA leaves out one ticket arrival, so the tile's finalize waits until its
(shortened) time limit passes.  The launch must then end by itself (every
wait bounded, every CTA winding down through the abort flag), report
TPL_DEVERR_TIMEOUT in the device error word, and leave nothing behind: the
next normal call on the same workspace equals a fresh one bit for bit."""
import time

import pytest
import torch

import synthetic_inputs as si

pytestmark = pytest.mark.gpu
tpl = pytest.importorskip("mlp_megatron_tp_layer_b300")

TIMEOUT_BIT = 0x1   # TPL_DEVERR_TIMEOUT


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.synchronize()
    tpl.device_status()
    yield
    tpl.test_fused_fault()
    torch.cuda.synchronize()
    assert tpl.device_status() == 0


SHAPE = dict(D=1024, F=2048, n_q=8, n_kv=2, hd=128, tp=2, L=2)
GRID = 148


def cta_with_work(M, G=GRID):
    """A CTA that holds units of a projection of M output rows whatever split
    the fused stack picks: a phase goes to m_tiles x s CTAs (every 128-row
    tile in s k-ranges, s >= 1), or is spread over the whole grid when it has
    at least G (m-tile, k-block) pairs (true of every phase used here), so
    CTAs 0 .. min(m_tiles, G) - 1 always have work; this is the last of them."""
    return min(-(-M // 128), G) - 1


_S = SHAPE
_QKV_ROWS = (_S["n_q"] + 2 * _S["n_kv"]) * _S["hd"]


def _stack(B, block):
    s = SHAPE
    layers = [si.layer_weights(s["D"], s["F"], s["n_q"], s["n_kv"], s["hd"], seed=31, layer=l, sigma=0.03,
                               device="cuda") for l in range(s["L"])]
    x = si.activations(B, s["D"], seed=31, device="cuda")

    def run():
        return tpl.tp_decoder_stack(x, layers, s["n_q"], s["n_kv"], s["hd"], s["tp"], path=tpl.PATH_FUSED,
                                    block=block)
    return run


# (cta, phase): phase 4 l + 1 + j is projection j of layer l in the block's order
@pytest.mark.parametrize("B,block,cta,phase", [
    (1, tpl.BLOCK_SERIAL, cta_with_work(_QKV_ROWS), 1),                  # QKV of layer 0
    (40, tpl.BLOCK_SERIAL, 0, 3),                                                       # gate/up of layer 0
    (1, tpl.BLOCK_SERIAL, cta_with_work(_S["D"]), 8),                     # down of layer 1
    (16, tpl.BLOCK_PARALLEL, cta_with_work(_S["D"]), 3),     # o_proj, finalized with down
])
def test_fused_stack_wait_runs_out_and_the_next_call_is_clean(B, block, cta, phase):
    run = _stack(B, block)
    ref = run()
    assert tpl.device_status() == 0
    tpl.test_fused_fault(cta, phase, 1_000_000)          # 1 ms limit
    t0 = time.perf_counter()
    run()                                                # the launch itself succeeds
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    flags = tpl.device_status()
    tpl.test_fused_fault()
    assert flags & TIMEOUT_BIT, f"expected a timed-out wait, flags={flags:#x}"
    assert dt < 1.0, f"the aborted launch took {dt:.3f} s"
    again = run()
    torch.cuda.synchronize()
    assert tpl.device_status() == 0
    assert torch.equal(again, ref), "the call after the aborted one differs from a fresh call"


def test_short_wait_limit_alone_changes_nothing():
    run = _stack(8, tpl.BLOCK_SERIAL)
    ref = run()
    tpl.test_fused_fault(-1, 1, 50_000_000)              # 50 ms, nothing left out
    y = run()
    torch.cuda.synchronize()
    assert tpl.device_status() == 0
    assert torch.equal(y, ref)


def test_phase_trace_is_only_in_the_instrumented_build():
    """The normal library records no phase stamps: the read is refused."""
    import ctypes
    buf = (ctypes.c_uint64 * 8)()
    st = tpl.lib.tpl_fused_trace_read(ctypes.cast(buf, ctypes.c_void_p), ctypes.sizeof(buf))
    if tpl.LIB_PATH.endswith("libtpl_trace.so"):
        assert st == 0
    else:
        assert tpl.STATUS[st] == "TPL_ERR_UNSUPPORTED"


# Repeated launches at the shapes where every k-block's activations arrive fast
# (small batches): a ring whose barrier phases could alias two rounds apart
# (a producer waiting for a release the consumer has already given twice)
# hangs only when a race is lost, so one launch proves little.  Every launch
# must end cleanly with the same bits.
@pytest.mark.parametrize("model,block,B,L,reps", [
    ("qwen", tpl.BLOCK_PARALLEL, 8, 28, 60),
    ("qwen", tpl.BLOCK_SERIAL, 1, 28, 60),
    ("llama", tpl.BLOCK_SERIAL, 1, 2, 30),
])
def test_fused_stack_repeated_launches_stay_clean(model, block, B, L, reps):
    cfg = si.QWEN_DECODE if model == "qwen" else si.LLAMA_DECODE
    D, F, n_q, n_kv, hd, tp = cfg["D"], cfg["F"], cfg["n_q"], cfg["n_kv"], cfg["head_dim"], cfg["tp"]
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix=model, device="cuda")
              for l in range(L)]
    x = si.activations(B, D, seed=5, name=f"{model}.rep{B}", device="cuda")
    ws = tpl.workspace(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp), "cuda")
    tpl.test_fused_fault(-1, 1, 200_000_000)           # a lost race ends in 0.2 s, not 2 s
    ref = None
    for r in range(reps):
        y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, ws=ws, path=tpl.PATH_FUSED, block=block)
        torch.cuda.synchronize()
        assert tpl.device_status() == 0, f"launch {r} timed out"
        if ref is None:
            ref = y.clone()
        else:
            assert torch.equal(y, ref), f"launch {r} differs from the first"
