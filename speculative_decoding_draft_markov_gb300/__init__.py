"""DSpark per-step speculative-decoding token path for GB300 (sm_103a).

The compute lives in the C-ABI library libdspark.so (CUDA kernels); `binding` is a thin
ctypes layer over it.  `inputs` holds the seeded synthetic input generators.
Importing the package loads nothing; the library is loaded on first use and a missing
or unbuilt library raises an error (there is no CPU fallback)."""
