"""Paged GQA decode / speculative-verify attention for one GB300 (sm_103a).

The product is the C-ABI library libpa (include/pa.h, sources in csrc/).
``binding`` exposes its entry points to Python under the same names;
``decode`` adds torch-side buffer management; ``workloads`` draws the seeded
synthetic inputs."""
