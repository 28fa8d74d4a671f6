"""Test-only CUDA library ``libgdnqat_testing.so`` (never loaded by the package itself).

- ``tc_selftest.cu``: one tcgen05 MMA on operands staged in the shared-memory layouts the
  chunk kernels use, read back from TMEM (the layout checks of test_gpu_tc_layouts.py).
- The two-kernel chunk forward (``chunk_prep.cu``, ``chunk_chain.cu``, ``tma_maps.cu`` of the
  product sources) compiled with ``GDN_WAIT_LIMIT=0``: every pipeline wait gives up at once, so
  each CTA takes its abort path (status word set, copies in flight drained with their own
  limits, TMEM freed). ``short_waits.cu`` exposes it as ``gdnqat_testing_split_fwd``.
- ``quotient_sweep.cu``: the standalone QDQ ops' corrected-reciprocal quotient against the IEEE
  divide over every significand of one operand (``gdnqat_testing_quotient_sweep``).
"""
import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libgdnqat_testing.so")
OBJ_DIR = os.path.join(HERE, "_lib", "_obj")

_lock = threading.Lock()
_lib = None


def _sources():
    from fp8_state_qat_gb300 import build as pb
    short = ["GDN_WAIT_LIMIT=0u"]
    return [os.path.join(HERE, "tc_selftest.cu"), os.path.join(HERE, "short_waits.cu"),
            os.path.join(HERE, "quotient_sweep.cu"),
            (os.path.join(pb.CSRC, "chunk_prep.cu"), short), (os.path.join(pb.CSRC, "chunk_chain.cu"), short),
            (os.path.join(pb.CSRC, "tma_maps.cu"), short)]


def build(force: bool = False) -> str:
    from fp8_state_qat_gb300 import build as pb
    srcs = _sources()
    deps = [s if isinstance(s, str) else s[0] for s in srcs] + pb.headers() + [__file__]
    if not force and pb.newer_than(LIB_PATH, deps):
        return LIB_PATH
    return pb.compile_library(srcs, LIB_PATH, OBJ_DIR)


def load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(LIB_PATH)
        return _lib
