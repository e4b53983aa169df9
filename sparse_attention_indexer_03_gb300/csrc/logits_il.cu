// The tensor-core logits kernel instantiated for K-caches in the interleaved
// layout (each token's 128 value bytes followed by its 4 scale bytes, as the
// aiter PR 4244 reproducer builds the cache), in a translation unit of its own
// so that it compiles in parallel with the page-split instantiations.
#define SAI_LOGITS_INTERLEAVED 1
#include "logits.cu"
