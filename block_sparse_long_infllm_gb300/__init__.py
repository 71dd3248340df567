"""InfLLM v2 block-sparse attention for GB300 (sm_103a).

`infllmv2` is the Python binding of the C-ABI library `libinfllmv2.so`
(kernel pooling, block selection, sparse prefill attention, decode and tree
verification); `synth` draws the seeded synthetic inputs.  Importing the
package loads nothing; the binding loads the CUDA library on first use and
raises if it is missing.
"""
__all__ = ["infllmv2", "synth"]
