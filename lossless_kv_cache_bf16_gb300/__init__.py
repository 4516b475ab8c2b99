"""SplitZip lossless KV-cache codec for GB300 (sm_103a).

``splitzip`` is the binding of the C ABI in ``include/splitzip.h``;
``workloads`` generates the seeded synthetic KV tensors; ``build`` compiles
the CUDA library in-tree.  Submodules are imported on demand so that the
generators and the build step load without the CUDA library.
"""
