"""Compressed sparse multi-query attention for GB300 (sm_103a).

The path (DeepSeek-V4-Flash attention as the "DS4 (DwarfStar 4)" page, Key
Techniques, "KV attention compression" describes it): a KV compressor that pools
each block of `ratio` tokens into one row, an indexer that keeps the top-k
compressed rows on ratio-4 layers, and multi-query attention as one softmax over
the raw 128-token window and the kept compressed rows.

`ds4a` is the thin ctypes binding of the C-ABI library libds4a.so (CUDA
kernels); `synth` draws seeded synthetic inputs; `schedule` holds the per-layer
configuration.  Importing this package loads nothing; the first call into
`ds4a` loads the library and raises if it has not been built.
"""
