"""GB300-native (sm_103a) lightning-indexer MQA-logits forward.

The compute path is a C-ABI CUDA library (include/dsa_indexer.h), loaded by
`infra_dsa_indexer_gb300.binding`; `synth` makes seeded inputs. Importing this
package loads nothing: the library is opened on the first binding call, and
that call raises if the library is missing.
"""
