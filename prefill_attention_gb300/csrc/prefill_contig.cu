// prefill_contig.cu -- the prefill kernels over a contiguous (stride-addressed) K/V cache, with
// and without an explicit mask: the kernel template of prefill.cu instantiated with
// CONTIG = true in a translation unit of its own.
#define ASTR_PREFILL_CONTIG_TU 1
#include "prefill.cu"
