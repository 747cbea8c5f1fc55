"""DFlash2 candidate-selector head on GB300 (sm_103a).

The compute path is the C-ABI library ``libdflash2.so`` (CUDA, built from
``csrc/``); :mod:`.dflash2` is its thin ctypes binding.  Importing this
package loads nothing; the binding loads the library on first use and raises
if it is missing (there is no CPU fallback).
"""
__all__ = ["dflash2", "synth"]
