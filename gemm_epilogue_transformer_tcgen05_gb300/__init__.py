"""GB300 (sm_103a) GEMM-epilogue programs: a tcgen05/TMEM GEMM mainloop whose output tile
stays on chip while a composable epilogue (row/column scaling, residual add, SwiGLU, RoPE,
partial reductions, precision cast) runs before the single store, and the Transformer
block chains built from it.  The compute lives in libcoda.so (include/coda.h); this
package is its ctypes binding (module ``coda``) and its build script (module ``build``).
"""
from . import coda  # noqa: F401

__all__ = ["coda"]
