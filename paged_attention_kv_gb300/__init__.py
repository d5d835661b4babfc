"""GB300-native paged-KV attention: slot mapping, KV write and attention over
a ragged continuous batch, as hand-written sm_103a CUDA behind a C ABI
(``include/pagedkv.h``). ``binding`` is the thin Python layer over it."""
