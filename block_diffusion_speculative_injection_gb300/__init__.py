"""DFlash speculate-and-verify on one GB300 (sm_103a): C-ABI library + binding.

``capi`` is the ctypes binding of include/dflash.h (same function names);
``engine`` is the host harness that uploads seeded weights and drives the
step loops; ``build`` compiles libdflash.so in this directory.  Importing the
package does not load the shared library; the first C call does, and fails
loudly if it has not been built.
"""
