"""Builds the exhaustive pin checker (oracle_pins.c + the oracle's C file)."""
import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))


def load() -> ctypes.CDLL:
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    srcs = [os.path.join(HERE, "oracle_pins.c"), os.path.join(ROOT, "oracle", "rlq_oracle.c")]
    so = os.path.join(out_dir, "libpins.so")
    if not os.path.exists(so) or any(os.path.getmtime(s) > os.path.getmtime(so) for s in srcs):
        tmp = so + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off",
                        "-fno-fast-math", "-fPIC", "-shared", *srcs, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, so)
    lib = ctypes.CDLL(so)
    lib.pin_encode_exhaustive.restype = ctypes.c_uint64
    lib.pin_encode_exhaustive.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.pin_quant_pairs.restype = ctypes.c_uint64
    lib.pin_quant_pairs.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    return lib
