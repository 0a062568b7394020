"""GB300-native query-aware (Quest-style) sparse decode attention.

The compute path is the CUDA library libsvquest.so (C ABI, include/svquest.h);
`query_aware_sparse_quest_gb300.binding` is its thin ctypes binding.  The
binding loads the library on first use and raises if it is missing: there is
no CPU fallback.  `synth` draws the seeded synthetic workloads.
"""
