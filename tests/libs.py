"""Test helper: build the package's CUDA libraries once if they are missing or stale."""
import glob
import os
import threading

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decode_verify_kda_gb300")
_lock = threading.Lock()


def ensure_built():
    from speculative_decode_verify_kda_gb300 import build
    libs = [os.path.join(build.LIB_DIR, n) for n in build.LIBS]
    srcs = glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    with _lock:
        if not all(os.path.exists(p) for p in libs) or \
                min(os.path.getmtime(p) for p in libs) < max(os.path.getmtime(s) for s in srcs):
            build.build()
    return libs
