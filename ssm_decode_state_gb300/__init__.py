"""ReplaySSM decode-state path for GB300 (sm_103a).

* ``replayssm``   -- ctypes binding of libreplayssm.so (the C ABI in
  include/replayssm.h); importing it fails if the library is not built.
* ``inputs``      -- seeded synthetic workloads (shapes and distributions).
* ``bytes_model`` -- algorithmic bytes per sequence and step of each path.
* ``build``       -- in-tree nvcc build of the library.

The package root imports nothing heavy, so the input generator and the
bytes model are usable without a GPU.
"""
