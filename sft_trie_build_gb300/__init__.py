"""Prefix-tree sequence packing and tree attention for GB300 (sm_103a).

``sft_trie_build_gb300.stp``       -- binding of libstp.so (include/stp.h)
``sft_trie_build_gb300.build``     -- builds libstp.so in-tree
``sft_trie_build_gb300.workloads`` -- seeded synthetic inputs
"""
