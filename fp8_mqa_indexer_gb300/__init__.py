"""GB300-native MQA logits scoring (the lightning-indexer step).

The compute runs in the CUDA library ``libmqa.so`` built from ``csrc/``; this
package is a thin binding over its C ABI (see ``include/mqa.h``).
"""
