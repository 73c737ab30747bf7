"""CPU oracle for EasySpec layer-parallel ("fuzzy") speculative decoding.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, deliberately
un-optimised restatement of what the method computes, written to check the
CUDA path against.  Only the test-suite, the package's ``smoke()`` self-check
and the benchmark's CPU-baseline leg may import it.  The product path (the
C-ABI library and its Python binding) never imports, calls or falls back to
anything in here.

Arithmetic is IEEE float64 (numpy) for every forward pass.  The steps where a
floating-point value decides an integer -- argmax, the accept test and the
integer-quantised categorical sampler -- take that decision in float32, the
precision the CUDA kernels use, so both sides decide on the same footing.

Sources (web pages describing the method):
  * "EasySpec: Layer-Parallel Speculative Decoding for Efficient Multi-GPU
    Utilization" -- OpenReview discussion page (paperhub.cn), author replies
    on Table 4 / Appendix B.1, Figure 1(b), Figure 2 and Table 3.
  * The same paper's arXiv abstract (index card page, 2502.02493).
  * The accept/resample rule is defined by two works that page lists among
    the paper's references: "Fast Inference from Transformers via Speculative
    Decoding" (Leviathan et al.) and "Accelerating Large Language Model
    Decoding with Speculative Sampling" (Chen et al.).

Parity status per function is stated in each module header.
"""
