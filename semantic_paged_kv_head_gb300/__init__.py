"""GB300-native IceCache decode-time path: DCI-tree page index, insertion,
prioritised page selection and paged sparse GQA attention.

``semantic_paged_kv_head_gb300.ice`` binds the CUDA library (``libice.so``);
``semantic_paged_kv_head_gb300.synth`` draws seeded synthetic inputs. Importing
the package itself loads nothing.
"""
