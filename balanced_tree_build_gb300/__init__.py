"""GB300-native builder for left-balanced, complete, level-order k-d trees."""
